"""GB300 (sm_103a) K-FAC preconditioning step.

The product is the C ABI of ``include/kfac.h`` implemented by the CUDA library
``libkfac_gb300.so`` (built in-tree by ``infra_fac_factors_gb300.build``).
``capi`` binds it with the same names; ``step.KFACStep`` runs a whole step
for a list of layers.
"""
from . import capi  # noqa: F401

__all__ = ["capi"]
