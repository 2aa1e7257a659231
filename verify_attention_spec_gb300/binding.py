"""Thin ctypes binding over libvas.so (declared in include/vas.h).

Argument marshalling only: torch tensors become device pointers and sizes, the current
torch stream becomes the cudaStream_t, and a non-zero status becomes a ``VasError``.
Every step of the computation runs in the library's CUDA kernels.  Importing this
module raises ``ImportError`` when the library has not been built; there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvas.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m verify_attention_spec_gb300._build` "
        "(or __graft_entry__.build()); this package has no CPU fallback")

_lib = ctypes.CDLL(LIB_PATH)

# status codes and device error bits (include/vas.h)
VAS_OK = 0
VAS_E_INVALID_ARG = -1
VAS_E_UNSUPPORTED = -2
VAS_E_WORKSPACE = -3
VAS_E_CUDA = -4
VAS_E_NOMEM = -5
VAS_E_NOT_FOUND = -6
VAS_E_EXISTS = -7
VAS_DEV_BAD_PAGE = 0x1
VAS_DEV_BAD_LENGTHS = 0x2
VAS_DEV_BAD_TOKEN = 0x4
VAS_DEV_EMPTY_ROW = 0x8
VAS_DEV_TIMEOUT = 0x10
VAS_DEV_BAD_TREE = 0x20
VAS_DEV_RESIDUAL_FALLBACK = 0x100
VAS_F32 = 0
VAS_BF16 = 1
VAS_FP8_E4M3 = 2
VAS_INT8 = 3

_c_void_p, _i32, _i64, _u32, _u64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                                  ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float,
                                                  ctypes.c_size_t)


class vas_attn_dims(ctypes.Structure):
    _fields_ = [("num_seqs", _i32), ("total_q_tokens", _i32), ("num_q_heads", _i32),
                ("num_kv_heads", _i32), ("head_dim", _i32), ("page_size", _i32),
                ("num_pages", _i32), ("max_pages_per_seq", _i32), ("kv_dtype", _i32),
                ("scale", _f32)]


_P_dims = ctypes.POINTER(vas_attn_dims)
_sig = {
    "paged_attn_workspace_size": ([_P_dims], _sz),
    "paged_attn_workspace_min": ([_P_dims], _sz),
    "paged_attn_fwd": ([_c_void_p] * 8 + [_P_dims, _c_void_p, _sz, _c_void_p], ctypes.c_int),
    "paged_attn_fwd_tree": ([_c_void_p] * 9 + [_P_dims, _c_void_p, _sz, _c_void_p], ctypes.c_int),
    "paged_attn_fwd_quant": ([_c_void_p] * 11 + [_P_dims, _c_void_p, _sz, _c_void_p], ctypes.c_int),
    "spec_verify": ([_c_void_p, _c_void_p, _c_void_p, _u64, _c_void_p, _c_void_p, _i32, _i32, _i32,
                     _c_void_p], ctypes.c_int),
    "spec_verify_tree": ([_c_void_p] * 4 + [_u64] + [_c_void_p] * 3 + [_i32, _i32, _i32, _c_void_p],
                         ctypes.c_int),
    "vas_last_device_error": ([ctypes.POINTER(_i32), _c_void_p], ctypes.c_int),
    "vas_philox4x32_10": ([_c_void_p, _u32, _u32, _c_void_p, _i64, _c_void_p], ctypes.c_int),
    "vas_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "vas_pool_create": ([_i32, _i32, _u64], _c_void_p),
    "vas_pool_destroy": ([_c_void_p], None),
    "vas_pool_free_pages": ([_c_void_p], _i32),
    "vas_pool_num_seqs": ([_c_void_p], _i32),
    "vas_pool_can_allocate": ([_c_void_p, _i32], ctypes.c_int),
    "vas_seq_pages_needed": ([_c_void_p, _i64, _i32], _i32),
    "vas_seq_len": ([_c_void_p, _i64], _i32),
    "vas_seq_admit": ([_c_void_p, _i64, _i32], ctypes.c_int),
    "vas_seq_grow": ([_c_void_p, _i64, _i32], ctypes.c_int),
    "vas_seq_rollback": ([_c_void_p, _i64, _i32], ctypes.c_int),
    "vas_seq_free": ([_c_void_p, _i64], ctypes.c_int),
    "vas_pool_preempt_newest": ([_c_void_p, ctypes.POINTER(_i64)], ctypes.c_int),
    "vas_seq_fork": ([_c_void_p, _i64, _i64, _i32], ctypes.c_int),
    "vas_page_refcount": ([_c_void_p, _i32], _i32),
    "vas_build_block_table": ([_c_void_p, _c_void_p, _i32, _c_void_p, _i32, _c_void_p], ctypes.c_int),
}
for _name, (_args, _res) in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


class VasError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {_lib.vas_status_string(status).decode()} ({status})")


def _check(fn: str, status: int) -> None:
    if status != VAS_OK:
        raise VasError(fn, status)


def _stream_ptr(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> ctypes.c_void_p:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


_KV_CODES = {torch.bfloat16: VAS_BF16, torch.float32: VAS_F32}


_QUANT_CODES = {"fp8": VAS_FP8_E4M3, "int8": VAS_INT8}


def attn_dims(q: torch.Tensor, k_pages: torch.Tensor, block_table: torch.Tensor,
              seq_lens: torch.Tensor, scale: float = 0.0, quant: Optional[str] = None) -> vas_attn_dims:
    """vas_attn_dims from tensor shapes: q [T, Hq, D], k_pages [num_pages, P, Hkv, D],
    block_table [B, max_pages], seq_lens [B].  quant: None (k_pages share q's dtype), or
    "fp8" / "int8" for a pool of 8-bit codes (uint8 tensors) with a bf16 q."""
    T, Hq, D = q.shape
    num_pages, P, Hkv, D2 = k_pages.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_pages differ")
    if quant is not None:
        if quant not in _QUANT_CODES or q.dtype != torch.bfloat16 or k_pages.dtype != torch.uint8:
            raise ValueError("a quantised pool is uint8 codes with a bf16 q")
        code = _QUANT_CODES[quant]
    else:
        if q.dtype not in _KV_CODES or k_pages.dtype != q.dtype:
            raise ValueError("q and k_pages must share a dtype in {bf16, fp32}")
        code = _KV_CODES[q.dtype]
    return vas_attn_dims(num_seqs=int(seq_lens.shape[0]), total_q_tokens=int(T), num_q_heads=int(Hq),
                         num_kv_heads=int(Hkv), head_dim=int(D), page_size=int(P),
                         num_pages=int(num_pages), max_pages_per_seq=int(block_table.shape[1]),
                         kv_dtype=code, scale=float(scale))


def paged_attn_workspace_size(dims: vas_attn_dims) -> int:
    return int(_lib.paged_attn_workspace_size(ctypes.byref(dims)))


def paged_attn_workspace_min(dims: vas_attn_dims) -> int:
    return int(_lib.paged_attn_workspace_min(ctypes.byref(dims)))


def alloc_workspace(dims: vas_attn_dims, device=None, nbytes: Optional[int] = None) -> torch.Tensor:
    n = paged_attn_workspace_size(dims) if nbytes is None else int(nbytes)
    if n <= 0:
        raise ValueError("invalid attention dims")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def paged_attn_fwd(q, k_pages, v_pages, block_table, seq_lens, query_lens, out, lse, workspace,
                   *, scale: float = 0.0, dims: Optional[vas_attn_dims] = None, stream=None) -> None:
    """Paged decode/verify attention (include/vas.h: paged_attn_fwd).  All tensors on the
    same CUDA device; out [T, Hq, D] (dtype of q) and lse fp32 [T, Hq] are written."""
    if dims is None:
        dims = attn_dims(q, k_pages, block_table, seq_lens, scale)
    st = _lib.paged_attn_fwd(
        _dev(q, "q"), _dev(k_pages, "k_pages", q.dtype), _dev(v_pages, "v_pages", q.dtype),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(query_lens, "query_lens", torch.int32), _dev(out, "out", q.dtype),
        _dev(lse, "lse", torch.float32), ctypes.byref(dims), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check("paged_attn_fwd", st)


def paged_attn_fwd_tree(q, k_pages, v_pages, block_table, seq_lens, query_lens, tree_mask, out,
                        lse, workspace, *, scale: float = 0.0, dims: Optional[vas_attn_dims] = None,
                        stream=None) -> None:
    """Draft-tree attention (include/vas.h: paged_attn_fwd_tree).  tree_mask [T] int64 (the
    bits of a uint64 per query token: its ancestors among its sequence's draft tokens)."""
    if dims is None:
        dims = attn_dims(q, k_pages, block_table, seq_lens, scale)
    if tree_mask.dtype not in (torch.int64, getattr(torch, "uint64", torch.int64)):
        raise ValueError("tree_mask must be a 64-bit integer tensor")
    if tree_mask.numel() != q.shape[0]:
        raise ValueError("tree_mask needs one word per query token")
    st = _lib.paged_attn_fwd_tree(
        _dev(q, "q"), _dev(k_pages, "k_pages", q.dtype), _dev(v_pages, "v_pages", q.dtype),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(query_lens, "query_lens", torch.int32), _dev(tree_mask, "tree_mask"),
        _dev(out, "out", q.dtype), _dev(lse, "lse", torch.float32), ctypes.byref(dims),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check("paged_attn_fwd_tree", st)


def paged_attn_fwd_quant(q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, query_lens,
                         out, lse, workspace, *, quant: str, tree_mask=None, scale: float = 0.0,
                         dims: Optional[vas_attn_dims] = None, stream=None) -> None:
    """Attention over a quantised pool (include/vas.h: paged_attn_fwd_quant).  k_pages /
    v_pages uint8 codes [num_pages, P, Hkv, D] ("fp8" E4M3 or "int8"); k_scale / v_scale
    fp32 [num_pages, Hkv, P]; q and out bf16; tree_mask as for paged_attn_fwd_tree or None."""
    if dims is None:
        dims = attn_dims(q, k_pages, block_table, seq_lens, scale, quant=quant)
    tm = ctypes.c_void_p(0)
    if tree_mask is not None:
        if tree_mask.numel() != q.shape[0]:
            raise ValueError("tree_mask needs one word per query token")
        tm = _dev(tree_mask, "tree_mask")
    st = _lib.paged_attn_fwd_quant(
        _dev(q, "q", torch.bfloat16), _dev(k_pages, "k_pages", torch.uint8),
        _dev(v_pages, "v_pages", torch.uint8), _dev(k_scale, "k_scale", torch.float32),
        _dev(v_scale, "v_scale", torch.float32), _dev(block_table, "block_table", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), _dev(query_lens, "query_lens", torch.int32), tm,
        _dev(out, "out", torch.bfloat16), _dev(lse, "lse", torch.float32), ctypes.byref(dims),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check("paged_attn_fwd_quant", st)


def spec_verify_tree(p, q, draft_tokens, parents, seed: int, accepted_len, out_tokens, path, *,
                     stream=None) -> None:
    """Verification of a draft tree (include/vas.h: spec_verify_tree).  p [B, n+1, V] fp32,
    q [B, n, V] fp32, draft_tokens and parents [B, n] int32 -> accepted_len [B],
    out_tokens [B, n+1], path [B, n]."""
    B, n1, V = p.shape
    st = _lib.spec_verify_tree(_dev(p, "p", torch.float32), _dev(q, "q", torch.float32),
                               _dev(draft_tokens, "draft_tokens", torch.int32),
                               _dev(parents, "parents", torch.int32),
                               ctypes.c_uint64(seed & (2**64 - 1)),
                               _dev(accepted_len, "accepted_len", torch.int32),
                               _dev(out_tokens, "out_tokens", torch.int32),
                               _dev(path, "path", torch.int32), B, n1 - 1, V, _stream_ptr(stream))
    _check("spec_verify_tree", st)


def spec_verify(p, q, draft_tokens, seed: int, accepted_len, out_tokens, *, stream=None) -> None:
    """Modified rejection sampling (include/vas.h: spec_verify).  p [B, k+1, V] fp32,
    q [B, k, V] fp32, draft_tokens [B, k] int32 -> accepted_len [B], out_tokens [B, k+1]."""
    B, k1, V = p.shape
    k = k1 - 1
    qp = _dev(q, "q", torch.float32) if k > 0 else ctypes.c_void_p(0)
    xp = _dev(draft_tokens, "draft_tokens", torch.int32) if k > 0 else ctypes.c_void_p(0)
    st = _lib.spec_verify(_dev(p, "p", torch.float32), qp, xp, ctypes.c_uint64(seed & (2**64 - 1)),
                          _dev(accepted_len, "accepted_len", torch.int32),
                          _dev(out_tokens, "out_tokens", torch.int32), B, k, V, _stream_ptr(stream))
    _check("spec_verify", st)


def vas_last_device_error(stream=None) -> int:
    bits = _i32(0)
    _check("vas_last_device_error", _lib.vas_last_device_error(ctypes.byref(bits), _stream_ptr(stream)))
    return int(bits.value)


def vas_philox4x32_10(counters: torch.Tensor, key0: int, key1: int, out: torch.Tensor, stream=None) -> None:
    n = counters.shape[0]
    _check("vas_philox4x32_10",
           _lib.vas_philox4x32_10(_dev(counters, "counters", torch.int32), key0 & 0xFFFFFFFF,
                                  key1 & 0xFFFFFFFF, _dev(out, "out", torch.int32), n,
                                  _stream_ptr(stream)))


def vas_status_string(status: int) -> str:
    return _lib.vas_status_string(status).decode()


class PagePool:
    """Host page allocator and block-table builder (include/vas.h: vas_pool_*)."""

    def __init__(self, num_pages: int, page_size: int, seed: int = 0):
        self._h = _lib.vas_pool_create(num_pages, page_size, ctypes.c_uint64(seed))
        if not self._h:
            raise ValueError("invalid pool arguments")
        self.num_pages, self.page_size = num_pages, page_size

    def close(self):
        if self._h:
            _lib.vas_pool_destroy(self._h)
            self._h = None

    __del__ = close

    @property
    def free_pages(self) -> int:
        return int(_lib.vas_pool_free_pages(self._h))

    @property
    def num_seqs(self) -> int:
        return int(_lib.vas_pool_num_seqs(self._h))

    def can_allocate(self, n_tokens: int) -> bool:
        return bool(_lib.vas_pool_can_allocate(self._h, n_tokens))

    def pages_needed(self, seq_id: int, n_tokens: int) -> int:
        r = int(_lib.vas_seq_pages_needed(self._h, seq_id, n_tokens))
        if r < 0:
            raise VasError("vas_seq_pages_needed", r)
        return r

    def seq_len(self, seq_id: int) -> int:
        r = int(_lib.vas_seq_len(self._h, seq_id))
        if r < 0:
            raise VasError("vas_seq_len", r)
        return r

    def admit(self, seq_id: int, n_tokens: int) -> int:
        return int(_lib.vas_seq_admit(self._h, seq_id, n_tokens))

    def grow(self, seq_id: int, n_tokens: int) -> int:
        return int(_lib.vas_seq_grow(self._h, seq_id, n_tokens))

    def rollback(self, seq_id: int, n_tokens: int) -> int:
        return int(_lib.vas_seq_rollback(self._h, seq_id, n_tokens))

    def free(self, seq_id: int) -> int:
        return int(_lib.vas_seq_free(self._h, seq_id))

    def fork(self, parent: int, child: int, n_tokens: int) -> int:
        return int(_lib.vas_seq_fork(self._h, parent, child, n_tokens))

    def refcount(self, page: int) -> int:
        return int(_lib.vas_page_refcount(self._h, page))

    def preempt_newest(self):
        v = _i64(0)
        st = int(_lib.vas_pool_preempt_newest(self._h, ctypes.byref(v)))
        return (st, int(v.value))

    def block_table(self, seq_ids, max_pages: int):
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        bt = np.empty((len(ids), max_pages), dtype=np.int32)
        lens = np.empty(len(ids), dtype=np.int32)
        st = _lib.vas_build_block_table(self._h, ids.ctypes.data_as(_c_void_p), len(ids),
                                        bt.ctypes.data_as(_c_void_p), max_pages,
                                        lens.ctypes.data_as(_c_void_p))
        _check("vas_build_block_table", st)
        return bt, lens
