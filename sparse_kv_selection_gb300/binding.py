"""ctypes binding of libprhs.so: argument marshalling only.

Every function here has the name of the C entry point it calls (without the
``prhs_`` prefix) and does no arithmetic of the method: it turns torch CUDA
tensors into device pointers, fills the ``prhs_kv`` descriptor, calls the C
function and raises ``PrhsError`` on a non-OK status. Torch only provides
device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

PRHS_OK, PRHS_EINVAL, PRHS_EUNSUPPORTED, PRHS_EWORKSPACE, PRHS_ECUDA, PRHS_EDEVICE = range(6)
PRHS_F32, PRHS_BF16 = 0, 1
DEV_TIMEOUT, DEV_BAD_INDEX, DEV_BAD_LEN, DEV_BAD_BLOCK, DEV_CAPACITY = 1, 2, 4, 8, 16

# Entry points declared in include/prhs.h, in declaration order.
EXPORTS = ["prhs_workspace_size", "prhs_workspace_init", "prhs_score_select", "prhs_retrieve",
           "prhs_score",
           "prhs_select", "prhs_cis_dilate",
           "prhs_sparse_attn", "prhs_sparse_attn_noalloc", "prhs_set_mass", "prhs_dense_attn",
           "prhs_decode_step", "prhs_append_kv", "prhs_selftest_wait_timeout", "prhs_last_error",
           "prhs_device_error_bits", "prhs_status_str", "prhs_last_message", "prhs_num_sms",
           "prhs_launch_count"]


class PrhsError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status}: {message}")
        self.status = status


class prhs_kv(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("B", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("d", ctypes.c_int), ("k", ctypes.c_void_p),
                ("v", ctypes.c_void_p), ("t_max", ctypes.c_int), ("seq_lens", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("block_size", ctypes.c_int),
                ("max_blocks", ctypes.c_int), ("num_blocks", ctypes.c_int)]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libprhs.so (fails loudly when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with python -m sparse_kv_selection_gb300.build")
    lib = ctypes.CDLL(path)
    P, I, F, D, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t
    KV = ctypes.POINTER(prhs_kv)
    sig = {
        "prhs_workspace_size": (Z, [KV, I]),
        "prhs_workspace_init": (I, [P, Z, P]),
        "prhs_score_select": (I, [KV, P, F, I, P, I, I, P, P, P, I, P, P, P, I, P, P, Z, P]),
        "prhs_retrieve": (I, [KV, P, F, I, P, I, I, P, P, P, I, P, P, P, I, P, P, P, P, Z, P]),
        "prhs_score": (I, [KV, P, F, P, P, Z, P]),
        "prhs_select": (I, [KV, P, I, P, I, I, P, P, P, I, P, P, P, I, P, P, Z, P]),
        "prhs_cis_dilate": (I, [KV, P, P, I, P, P, I, I, I, I, D, I, P, P, P, I, P, P]),
        "prhs_sparse_attn": (I, [KV, P, F, P, P, I, P, P, P, Z, P]),
        "prhs_sparse_attn_noalloc": (I, [KV, P, F, P, P, I, P, P, P]),
        "prhs_set_mass": (I, [KV, P, F, P, P, I, P, P, Z, P]),
        "prhs_dense_attn": (I, [KV, P, F, P, P, P, Z, P]),
        "prhs_decode_step": (I, [KV, P, P, F, I, P, I, I, I, I, D, I, P, P, P, I, P, P, P, I, P, P, P, P,
                                 P, Z, P]),
        "prhs_append_kv": (I, [KV, P, P, P]),
        "prhs_selftest_wait_timeout": (I, [ctypes.c_uint, P]),
        "prhs_last_error": (I, []),
        "prhs_device_error_bits": (ctypes.c_uint, []),
        "prhs_launch_count": (ctypes.c_ulonglong, []),
        "prhs_status_str": (ctypes.c_char_p, [I]),
        "prhs_last_message": (ctypes.c_char_p, []),
        "prhs_num_sms": (I, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str) -> None:
    if status != PRHS_OK:
        raise PrhsError(status, where, load().prhs_last_message().decode())


class KVCache:
    """Device-resident KV cache plus the descriptor the C ABI takes.

    ``k``/``v`` are contiguous [B][Hkv][t_max][d] or paged
    [num_blocks][Hkv][block_size][d] tensors of dtype float32 or bfloat16;
    ``seq_lens`` int32 [B]; ``block_table`` int32 [B][max_blocks] or None.
    """

    def __init__(self, k, v, seq_lens, Hq, block_table=None, block_size=16):
        assert k.is_cuda and v.is_cuda and k.shape == v.shape
        self.k, self.v = k.contiguous(), v.contiguous()
        self.seq_lens = seq_lens.to(torch.int32).contiguous()
        self.block_table = None if block_table is None else block_table.to(torch.int32).contiguous()
        self.desc = prhs_kv()
        d = self.desc
        d.dtype = PRHS_BF16 if k.dtype == torch.bfloat16 else PRHS_F32
        if k.dtype not in (torch.bfloat16, torch.float32):
            raise ValueError("cache dtype must be float32 or bfloat16")
        d.Hq = Hq
        d.d = k.shape[-1]
        d.Hkv = k.shape[1]
        d.k, d.v = _ptr(self.k), _ptr(self.v)
        d.seq_lens = _ptr(self.seq_lens)
        if self.block_table is None:
            d.B, d.t_max = k.shape[0], k.shape[2]
            d.block_table, d.block_size, d.max_blocks, d.num_blocks = None, 0, 0, 0
        else:
            d.B = self.block_table.shape[0]
            d.t_max = 0
            d.block_table = _ptr(self.block_table)
            d.block_size = k.shape[2]
            d.max_blocks = self.block_table.shape[1]
            d.num_blocks = k.shape[0]

    @property
    def B(self):
        return self.desc.B

    @property
    def Hq(self):
        return self.desc.Hq

    @property
    def t_max(self):
        d = self.desc
        return d.t_max if self.block_table is None else d.max_blocks * d.block_size

    def ref(self):
        return ctypes.byref(self.desc)


def workspace_size(kv: KVCache, cap: int = 0) -> int:
    n = load().prhs_workspace_size(kv.ref(), cap)
    if n == 0:
        raise PrhsError(PRHS_EINVAL, "workspace_size", load().prhs_last_message().decode())
    return n


def workspace_init(ws, stream=None) -> None:
    _check(load().prhs_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "workspace_init")


def make_workspace(kv: KVCache, cap: int = 0, stream=None):
    """Allocate (through torch) and zero a workspace for this cache."""
    n = workspace_size(kv, cap)
    ws = torch.empty(n, dtype=torch.uint8, device=kv.k.device)
    workspace_init(ws, stream)
    return ws


def score_select(kv, q, scale, N, idx, n_sel, delta, ws, *, n_budget=None, head_skip=None,
                 anchor_idx=None, anchor_n=None, q_anchor=None, n_sink=0, window=0,
                 stream=None) -> None:
    cap = idx.shape[-1]
    acap = anchor_idx.shape[-1] if anchor_idx is not None else 0
    _check(load().prhs_score_select(kv.ref(), _ptr(q), float(scale), int(N), _ptr(n_budget),
                                    int(n_sink), int(window),
                                    _ptr(head_skip), _ptr(idx), _ptr(n_sel), cap, _ptr(delta),
                                    _ptr(anchor_idx), _ptr(anchor_n), acap, _ptr(q_anchor),
                                    _ptr(ws), ws.numel(), _stream(stream)), "score_select")


def retrieve(kv, q, scale, N, idx, n_sel, delta, out, lse, ws, *, n_budget=None, head_skip=None,
             anchor_idx=None, anchor_n=None, q_anchor=None, n_sink=0, window=0,
             stream=None) -> None:
    """Top-N set, delta and the attention over the set for the heads not
    flagged in head_skip (prhs_retrieve); out [B][Hq][d] and lse [B][Hq] fp32."""
    cap = idx.shape[-1]
    acap = anchor_idx.shape[-1] if anchor_idx is not None else 0
    _check(load().prhs_retrieve(kv.ref(), _ptr(q), float(scale), int(N), _ptr(n_budget),
                                int(n_sink), int(window),
                                _ptr(head_skip), _ptr(idx), _ptr(n_sel), cap, _ptr(delta),
                                _ptr(anchor_idx), _ptr(anchor_n), acap, _ptr(q_anchor),
                                _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)),
           "retrieve")


def score(kv, q, scale, ws, *, head_skip=None, stream=None) -> None:
    _check(load().prhs_score(kv.ref(), _ptr(q), float(scale), _ptr(head_skip), _ptr(ws),
                             ws.numel(), _stream(stream)), "score")


def select(kv, q, N, idx, n_sel, delta, ws, *, n_budget=None, head_skip=None, anchor_idx=None,
           anchor_n=None, q_anchor=None, n_sink=0, window=0, stream=None) -> None:
    cap = idx.shape[-1]
    acap = anchor_idx.shape[-1] if anchor_idx is not None else 0
    _check(load().prhs_select(kv.ref(), _ptr(q), int(N), _ptr(n_budget), int(n_sink), int(window),
                              _ptr(head_skip),
                              _ptr(idx), _ptr(n_sel), cap, _ptr(delta), _ptr(anchor_idx),
                              _ptr(anchor_n), acap, _ptr(q_anchor), _ptr(ws), ws.numel(),
                              _stream(stream)), "select")


def cis_dilate(kv, anchor_idx, anchor_n, q, q_anchor, w, tau, idx, n_sel, reuse, *, max_run=0,
               anchor_age=None, n_sink=0, window=0, n_den=0, stream=None) -> None:
    _check(load().prhs_cis_dilate(kv.ref(), _ptr(anchor_idx), _ptr(anchor_n), anchor_idx.shape[-1],
                                  _ptr(q), _ptr(q_anchor), int(w), int(n_den), int(n_sink),
                                  int(window), float(tau), int(max_run),
                                  _ptr(anchor_age), _ptr(idx), _ptr(n_sel), idx.shape[-1],
                                  _ptr(reuse), _stream(stream)), "cis_dilate")


def set_mass(kv, q, scale, idx, n_sel, delta, ws, stream=None) -> None:
    """Dropped attention mass of the given sets under q (prhs_set_mass)."""
    _check(load().prhs_set_mass(kv.ref(), _ptr(q), float(scale), _ptr(idx), _ptr(n_sel),
                                idx.shape[-1], _ptr(delta), _ptr(ws), ws.numel(), _stream(stream)),
           "set_mass")


def sparse_attn(kv, q, scale, idx, n_sel, out, lse, ws, stream=None) -> None:
    _check(load().prhs_sparse_attn(kv.ref(), _ptr(q), float(scale), _ptr(idx), _ptr(n_sel),
                                   idx.shape[-1], _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                   _stream(stream)), "sparse_attn")


def sparse_attn_noalloc(kv, q, scale, idx, n_sel, out, lse, stream=None) -> None:
    """prhs_sparse_attn without a workspace (fixed in-library scratch)."""
    _check(load().prhs_sparse_attn_noalloc(kv.ref(), _ptr(q), float(scale), _ptr(idx),
                                           _ptr(n_sel), idx.shape[-1], _ptr(out), _ptr(lse),
                                           _stream(stream)), "sparse_attn_noalloc")


def dense_attn(kv, q, scale, out, lse, ws, stream=None) -> None:
    _check(load().prhs_dense_attn(kv.ref(), _ptr(q), float(scale), _ptr(out), _ptr(lse),
                                  _ptr(ws), ws.numel(), _stream(stream)), "dense_attn")


def decode_step(kv, q, scale, N, w, tau, anchor_idx, anchor_n, q_anchor, idx, n_sel, reuse, delta,
                out, lse, ws, *, n_budget=None, max_run=0, anchor_age=None, n_sink=0, window=0,
                n_den=0, gate=None, stream=None) -> None:
    _check(load().prhs_decode_step(kv.ref(), _ptr(q), _ptr(gate), float(scale), int(N),
                                   _ptr(n_budget), int(n_sink), int(window), int(w), int(n_den),
                                   float(tau), int(max_run), _ptr(anchor_age), _ptr(anchor_idx),
                                   _ptr(anchor_n),
                                   anchor_idx.shape[-1], _ptr(q_anchor), _ptr(idx), _ptr(n_sel),
                                   idx.shape[-1], _ptr(reuse), _ptr(delta), _ptr(out), _ptr(lse),
                                   _ptr(ws), ws.numel(), _stream(stream)), "decode_step")


def append_kv(kv, k_new, v_new, stream=None) -> None:
    """Write one key and value row per (sequence, KV head) at each
    sequence's current length and advance kv.seq_lens (prhs_append_kv)."""
    _check(load().prhs_append_kv(kv.ref(), _ptr(k_new), _ptr(v_new), _stream(stream)), "append_kv")


def selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Run the bounded-wait self-test kernel (prhs_selftest_wait_timeout): its
    wait runs out after limit_us and sets DEV_TIMEOUT in the error word."""
    _check(load().prhs_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "selftest_wait_timeout")


def last_error() -> int:
    """Synchronise, read and clear the device error word; return its bits."""
    lib = load()
    s = lib.prhs_last_error()
    if s == PRHS_EDEVICE:
        return int(lib.prhs_device_error_bits())
    _check(s, "last_error")
    return 0


def num_sms() -> int:
    return int(load().prhs_num_sms())


def launch_count() -> int:
    """Kernels the library has issued since it was loaded (prhs_launch_count)."""
    return int(load().prhs_launch_count())


def status_str(s: int) -> str:
    return load().prhs_status_str(s).decode()
