"""Absorbed multi-head latent attention (MLA) decode for GB300 (sm_103a).

The compute path is the C-ABI library ``libmla_decode.so`` built from
``csrc/``; ``binding`` marshals torch tensors into it.  Importing this package
does not load the library: ``binding`` does, and raises if it is missing.
"""
__all__ = ["workloads", "binding"]
