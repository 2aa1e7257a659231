"""CPU oracle for paged decode/verify attention and speculative rejection sampling.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product library (``verify_attention_spec_gb300``) never imports it, links it or
falls back to it; the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, OpenMP over independent
rows); this module only builds it with gcc and marshals numpy arrays through ctypes.
Every function cites the passage it follows in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2
Q_E4M3, Q_INT8 = 0, 1  # quantised KV formats (oracle.c: oracle_dequant_kv)
OK, E_ARG, E_PAGE, E_LEN, E_TOKEN, E_DIST = 0, -1, -2, -3, -4, -5

# Decisions whose uniform lies within this distance of its threshold are flagged
# (the tolerance the spec states for accepted lengths and emitted tokens).
FLAG_WINDOW = 1e-6


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (portable flags, no FMA contraction)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    i32, i64, u64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
    lib.oracle_paged_attn.argtypes = [P, P, P, i32, P, P, P, i32, i32, i32, i32, i32, i32,
                                      i32, dbl, P, P]
    lib.oracle_paged_attn.restype = i32
    lib.oracle_paged_attn_tree.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, i32, i32, i32,
                                           i32, i32, dbl, P, P]
    lib.oracle_paged_attn_tree.restype = i32
    lib.oracle_dequant_kv.argtypes = [P, P, i32, i64, i32, i32, i32, P]
    lib.oracle_dequant_kv.restype = i32
    lib.oracle_philox4x32_10.argtypes = [P, P, P]
    lib.oracle_philox4x32_10.restype = None
    lib.oracle_philox4x32_10_many.argtypes = [P, i64, P, P]
    lib.oracle_philox4x32_10_many.restype = None
    lib.oracle_uniforms.argtypes = [u64, i32, i32, P, P]
    lib.oracle_uniforms.restype = None
    lib.oracle_spec_verify_given_uniforms.argtypes = [P, P, P, P, P, i32, i32, i32, dbl, P, P,
                                                      P, P, P]
    lib.oracle_spec_verify_given_uniforms.restype = i32
    lib.oracle_spec_verify.argtypes = [P, P, P, u64, i32, i32, i32, dbl, P, P, P, P, P]
    lib.oracle_spec_verify.restype = i32
    lib.oracle_spec_verify_tree_given_uniforms.argtypes = [P, P, P, P, P, P, i32, i32, i32, dbl,
                                                           P, P, P, P, P, P]
    lib.oracle_spec_verify_tree_given_uniforms.restype = i32
    lib.oracle_spec_verify_tree.argtypes = [P, P, P, P, u64, i32, i32, i32, dbl, P, P, P, P, P, P]
    lib.oracle_spec_verify_tree.restype = i32
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i32
    lib.oracle_set_num_threads.argtypes = [i32]
    lib.oracle_set_num_threads.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on (for timing)."""
    _load().oracle_set_num_threads(int(n))


def _as_storage(x: np.ndarray, dtype_code: int) -> np.ndarray:
    if dtype_code == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype_code == BF16:
        return np.ascontiguousarray(x, dtype=np.uint16)  # raw bf16 bit patterns
    return np.ascontiguousarray(x, dtype=np.float64)


def paged_attn(q, k_pages, v_pages, block_table, seq_lens, query_lens, *, dtype_code: int,
               scale: float | None = None, parents=None):
    """Float64 paged attention (oracle.c: oracle_paged_attn, oracle_paged_attn_tree).

    q: [total_q_tokens, Hq, D]; k_pages/v_pages: [num_pages, page_size, Hkv, D], given as
    float32, raw bf16 bits (uint16) or float64 according to ``dtype_code``.
    parents: optional int32 [total_q_tokens], a draft tree (each query token's parent
    among its sequence's query tokens, -1 for a root); None is the causal window.
    Returns (out float64 [total_q_tokens, Hq, D], lse float64 [total_q_tokens, Hq]).
    """
    lib = _load()
    q = _as_storage(q, dtype_code)
    k_pages = _as_storage(k_pages, dtype_code)
    v_pages = _as_storage(v_pages, dtype_code)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ql = np.ascontiguousarray(query_lens, dtype=np.int32)
    T, Hq, D = q.shape
    num_pages, page_size, Hkv, D2 = k_pages.shape
    assert D2 == D and v_pages.shape == k_pages.shape
    B = sl.shape[0]
    maxp = bt.shape[1] if bt.ndim == 2 else 0
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    lse = np.zeros((T, Hq), dtype=np.float64)
    if parents is None:
        rc = lib.oracle_paged_attn(_ptr(q), _ptr(k_pages), _ptr(v_pages), dtype_code, _ptr(bt),
                                   _ptr(sl), _ptr(ql), B, Hq, Hkv, D, page_size, num_pages,
                                   maxp, float(scale), _ptr(out), _ptr(lse))
    else:
        par = np.ascontiguousarray(parents, dtype=np.int32)
        assert par.shape == (T,)
        rc = lib.oracle_paged_attn_tree(_ptr(q), _ptr(k_pages), _ptr(v_pages), dtype_code,
                                        _ptr(bt), _ptr(sl), _ptr(ql), _ptr(par), B, Hq, Hkv, D,
                                        page_size, num_pages, maxp, float(scale), _ptr(out),
                                        _ptr(lse))
    if rc != OK:
        raise ValueError(f"oracle_paged_attn rejected its arguments (code {rc})")
    return out, lse


def dequant_kv(codes, scales, fmt: int) -> np.ndarray:
    """Decode a quantised page pool (oracle.c: oracle_dequant_kv).  codes uint8
    [num_pages, P, Hkv, D]; scales float32 [num_pages, Hkv, P].  Returns float64
    [num_pages, P, Hkv, D]."""
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    n, P, Hkv, D = c.shape
    assert sc.shape == (n, Hkv, P)
    out = np.empty(c.shape, dtype=np.float64)
    rc = lib.oracle_dequant_kv(_ptr(c), _ptr(sc), int(fmt), n, P, Hkv, D, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_dequant_kv rejected its arguments (code {rc})")
    return out


def paged_attn_quant(q_bf16_bits, k_codes, v_codes, k_scale, v_scale, block_table, seq_lens,
                     query_lens, *, fmt: int, scale: float | None = None, parents=None):
    """Attention over a quantised pool: the pool decoded exactly (dequant_kv), then the
    float64 attention of paged_attn.  q is given as raw bf16 bits [T, Hq, D]."""
    qf = (np.ascontiguousarray(q_bf16_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return paged_attn(qf.astype(np.float64), dequant_kv(k_codes, k_scale, fmt),
                      dequant_kv(v_codes, v_scale, fmt), block_table, seq_lens, query_lens,
                      dtype_code=F64, scale=scale, parents=parents)


def philox4x32_10(counters: np.ndarray, key) -> np.ndarray:
    """Philox4x32-10 of each 128-bit counter row [n, 4] (uint32) under key (k0, k1)."""
    lib = _load()
    ctr = np.ascontiguousarray(counters, dtype=np.uint32).reshape(-1, 4)
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros_like(ctr)
    lib.oracle_philox4x32_10_many(_ptr(ctr), ctr.shape[0], _ptr(k), _ptr(out))
    return out


def uniforms(seed: int, B: int, k: int):
    """The uniforms the rule consumes: r [B, k] and s [B, k+1] (oracle.c: oracle_uniforms)."""
    lib = _load()
    r = np.zeros((B, max(k, 0)), dtype=np.float64)
    s = np.zeros((B, k + 1), dtype=np.float64)
    lib.oracle_uniforms(ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), B, k, _ptr(r), _ptr(s))
    return r, s


class VerifyResult:
    def __init__(self, accepted_len, out_tokens, margin, flag_pos, fallback, status, path=None):
        self.accepted_len = accepted_len
        self.out_tokens = out_tokens
        self.margin = margin
        self.flag_pos = flag_pos
        self.fallback = fallback
        self.status = status
        self.path = path  # tree verification: the accepted nodes


def _verify_buffers(B, k):
    return (np.zeros(B, dtype=np.int32), np.zeros((B, k + 1), dtype=np.int32),
            np.zeros(B, dtype=np.float64), np.zeros(B, dtype=np.int32),
            np.zeros(B, dtype=np.int32))


def spec_verify_given_uniforms(p, q, draft_tokens, r, s, flag_window: float = FLAG_WINDOW):
    """Modified rejection sampling with explicit uniforms
    (oracle.c: oracle_spec_verify_given_uniforms).  p [B,k+1,V], q [B,k,V] float32."""
    lib = _load()
    p = np.ascontiguousarray(p, dtype=np.float32)
    B, k1, V = p.shape
    k = k1 - 1
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(B, k, V)
    x = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, k)
    r = np.ascontiguousarray(r, dtype=np.float64).reshape(B, k)
    s = np.ascontiguousarray(s, dtype=np.float64).reshape(B, k + 1)
    acc, out, mg, fp, fb = _verify_buffers(B, k)
    rc = lib.oracle_spec_verify_given_uniforms(_ptr(p), _ptr(q), _ptr(x), _ptr(r), _ptr(s), B,
                                               k, V, float(flag_window), _ptr(acc), _ptr(out),
                                               _ptr(mg), _ptr(fp), _ptr(fb))
    return VerifyResult(acc, out, mg, fp, fb, rc)


def spec_verify(p, q, draft_tokens, seed: int, flag_window: float = FLAG_WINDOW):
    """Philox uniforms + modified rejection sampling (oracle.c: oracle_spec_verify)."""
    lib = _load()
    p = np.ascontiguousarray(p, dtype=np.float32)
    B, k1, V = p.shape
    k = k1 - 1
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(B, k, V)
    x = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, k)
    acc, out, mg, fp, fb = _verify_buffers(B, k)
    rc = lib.oracle_spec_verify(_ptr(p), _ptr(q), _ptr(x),
                                ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), B, k, V,
                                float(flag_window), _ptr(acc), _ptr(out), _ptr(mg), _ptr(fp),
                                _ptr(fb))
    return VerifyResult(acc, out, mg, fp, fb, rc)


def _tree_args(p, q, draft_tokens, parents):
    p = np.ascontiguousarray(p, dtype=np.float32)
    B, n1, V = p.shape
    n = n1 - 1
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(B, n, V)
    x = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, n)
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, n)
    acc, out, mg, fp, fb = _verify_buffers(B, n)
    path = np.zeros((B, n), dtype=np.int32)
    return p, q, x, par, B, n, V, acc, out, mg, fp, fb, path


def spec_verify_tree_given_uniforms(p, q, draft_tokens, parents, r, s,
                                    flag_window: float = FLAG_WINDOW):
    """Verification of a draft tree with explicit uniforms
    (oracle.c: oracle_spec_verify_tree_given_uniforms).  p [B, n+1, V], q [B, n, V],
    draft_tokens and parents [B, n] (parents[b, i]: the parent node of node i + 1, 0 for
    the root); r [B, n], s [B, n+1]."""
    lib = _load()
    p, q, x, par, B, n, V, acc, out, mg, fp, fb, path = _tree_args(p, q, draft_tokens, parents)
    r = np.ascontiguousarray(r, dtype=np.float64).reshape(B, n)
    s = np.ascontiguousarray(s, dtype=np.float64).reshape(B, n + 1)
    rc = lib.oracle_spec_verify_tree_given_uniforms(
        _ptr(p), _ptr(q), _ptr(x), _ptr(par), _ptr(r), _ptr(s), B, n, V, float(flag_window),
        _ptr(acc), _ptr(out), _ptr(path), _ptr(mg), _ptr(fp), _ptr(fb))
    return VerifyResult(acc, out, mg, fp, fb, rc, path)


def spec_verify_tree(p, q, draft_tokens, parents, seed: int, flag_window: float = FLAG_WINDOW):
    """Philox uniforms + the tree walk (oracle.c: oracle_spec_verify_tree)."""
    lib = _load()
    p, q, x, par, B, n, V, acc, out, mg, fp, fb, path = _tree_args(p, q, draft_tokens, parents)
    rc = lib.oracle_spec_verify_tree(_ptr(p), _ptr(q), _ptr(x), _ptr(par),
                                     ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), B, n, V,
                                     float(flag_window), _ptr(acc), _ptr(out), _ptr(path),
                                     _ptr(mg), _ptr(fp), _ptr(fb))
    return VerifyResult(acc, out, mg, fp, fb, rc, path)
