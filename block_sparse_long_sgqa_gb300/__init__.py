"""Block-wise Sparse GQA prefill for GB300 (sm_103a).

The compute path lives in the CUDA library ``libsgqa.so`` (C ABI declared in
``include/sgqa.h``); ``block_sparse_long_sgqa_gb300.sgqa`` is its thin ctypes
binding.  ``block_sparse_long_sgqa_gb300.synth`` draws the seeded synthetic
workloads.  Submodules load lazily so that the input generator can be used on
hosts without a GPU.
"""
__all__ = ["sgqa", "synth"]


def __getattr__(name):
    if name in __all__:
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
