"""GB300-native Pre-hoc Sparsity (PrHS) sparse-decode path.

The compute lives in ``libprhs.so`` (hand-written sm_103a CUDA behind a C
ABI, declared in ``include/prhs.h``); ``binding`` marshals torch tensors
into it and ``decoder`` keeps the per-head CIS anchor state of a decode
sequence. Nothing here falls back to host code: without the built library
every call raises.
"""
from .binding import (KVCache, PrhsError, cis_dilate, decode_step, dense_attn, last_error,
                      load, make_workspace, num_sms, retrieve, score_select, set_mass,
                      sparse_attn, workspace_init, workspace_size)
from .decoder import SparseDecoder

__all__ = ["KVCache", "PrhsError", "SparseDecoder", "cis_dilate", "decode_step", "dense_attn",
           "last_error", "load", "make_workspace", "num_sms", "retrieve", "score_select",
           "set_mass", "sparse_attn", "workspace_init", "workspace_size"]
