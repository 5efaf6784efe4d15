"""Truly sparse linear layer for NVIDIA GB300 (sm_103a).

The weight W (out x in) is stored only as its non-zeros, in a COO triple.  The
CUDA library ``libsnk`` computes the forward SpMM, the transposed SpMM for the
input gradient, the weight gradient on the support (SDDMM) and the in-place
prune/regrow restructure.  This package holds the C-ABI binding to it
(``binding``), a torch.nn front end with autograd and the SET schedule
(``module``), and the seeded synthetic input generators (``synth``).  The
binding is loaded on first use, so importing the package (or ``synth``) does
not touch the GPU.
"""
import importlib

__all__ = ["synth", "binding", "module"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
