"""Seeded synthetic workloads for the paged decode/verify attention + spec_verify path.

This module only *generates inputs*: sequence lengths, permuted page pools, block
tables, Q/K/V values and the target/draft distributions with their draft tokens.  It
holds none of the method's arithmetic (no attention, no acceptance test, no residual,
no draw from a residual); both the CUDA path and the CPU oracle consume what it makes.

Five workloads (named by what they are, counted from 0):

* ``tiny``      - fp32, 4 sequences of context {17, 40, 63, 100} with query lengths
                  {1, 4, 1, 4}; 4 query / 2 KV heads, head_dim 64, page 16, pages at
                  random permuted slots of a 64-page pool; spec_verify over vocab 128
                  for the two k=3 sequences.
* ``decode64``  - 64 decode sequences, Llama-3-8B attention shape (32/8 heads, d=128),
                  bf16, page 16, log-normal lengths (median 1024, sigma 1.0) clamped to
                  [128, 8192].
* ``verify32``  - 32 sequences with k=4 drafts (5 query tokens), lengths uniform in
                  [512, 4096], same 32/8/128 bf16 layout, page 16; spec_verify over
                  vocab 128256, Philox seed 1234.
* ``mixed272``  - 256 decode + 16 verify (k=7) sequences, 32/8/128 bf16, page 16,
                  Pareto lengths (alpha 1.5, minimum 64) capped at 32768; spec_verify over
                  vocab 32000.
* ``stress70b`` - 512 sequences, 70B attention shape (64/8 heads, d=128), bf16, page 32,
                  log-normal lengths (median 2048, sigma 1.2) clamped to [256, 32768];
                  448 decode + 64 verify with k=4; spec_verify over vocab 128256, seed 99.

and beyond them, for chunked prefill:

* ``prefill8``  - 8 sequences of context 4096, each bringing a 1024-token prompt chunk
                  (query length 1024, causal within the chunk), 70B attention shape,
                  bf16, page 32; no spec_verify;

for prefix sharing, ``shared70b``: the 70B batch with a 2048-token system prompt in
front of every sequence, its 64 pages shared by groups of 8 consecutive sequences;

and for quantised KV pages, the 70B batch and decode64 with the same lengths, seeds and
spec_verify, their K/V stored as FP8 E4M3 or INT8 codes with one fp32 scale per
(token, KV head) for K and one for V (``stress70b_fp8``, ``stress70b_int8``,
``decode64_fp8``, ``decode64_int8``).  The codes come from the same N(0, 1) draws:
scale = max |x| over the head's D values / 448 (E4M3) or / 127 (INT8), code = x / scale
rounded to nearest (E4M3 by torch's float8_e4m3fn conversion).

Distributions (the pages leave them open; the plainest readings are taken): N(0, s) means
standard deviation s; log-normal L = round(exp(ln median + sigma z)); Pareto
L = floor(x_min (1 - U)^(-1/alpha)); uniform integers inclusive; p = softmax(logits),
logits ~ N(0, s_p); q = softmax(logits + N(0, s_q) noise); drafts x_i ~ q_i.  The page
pool is "sized for the total" (exactly sum ceil(L_i / P) pages) unless a pool size is
given; pages are handed to sequences from a seeded random permutation.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

F32 = "f32"
BF16 = "bf16"
FP8 = "fp8"    # K/V pages as FP8 E4M3 codes with a scale per (token, KV head); Q bf16
INT8 = "int8"  # K/V pages as INT8 codes with a scale per (token, KV head); Q bf16
QUANTIZED = (FP8, INT8)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_dtype: str
    length_law: str            # "fixed" | "lognormal" | "uniform" | "pareto"
    length_args: tuple
    num_seqs: int
    num_verify: int            # how many of num_seqs are verify sequences
    k: int                     # drafts per verify sequence (query length k + 1)
    vocab: int                 # 0: no spec_verify in this workload
    p_logit_std: float = 3.0
    q_noise_std: float = 1.5
    pool_pages: Optional[int] = None     # None: sized for the total
    fixed_lens: Optional[tuple] = None
    fixed_qlens: Optional[tuple] = None
    prefix_tokens: int = 0     # a shared prefix (whole pages) added to every sequence ...
    prefix_group: int = 0      # ... shared by consecutive groups of this many sequences
    tree: bool = False         # the verify windows are draft trees (k nodes under the root)


WORKLOADS = {
    "tiny": Workload("tiny", 0, 4, 2, 64, 16, F32, "fixed", (), 4, 2, 3, 128,
                     p_logit_std=2.0, q_noise_std=1.0, pool_pages=64,
                     fixed_lens=(17, 40, 63, 100), fixed_qlens=(1, 4, 1, 4)),
    "decode64": Workload("decode64", 1, 32, 8, 128, 16, BF16, "lognormal", (1024.0, 1.0, 128, 8192),
                         64, 0, 0, 0),
    "verify32": Workload("verify32", 1234, 32, 8, 128, 16, BF16, "uniform", (512, 4096),
                         32, 32, 4, 128256),
    "mixed272": Workload("mixed272", 3, 32, 8, 128, 16, BF16, "pareto", (1.5, 64, 32768),
                         272, 16, 7, 32000),
    "stress70b": Workload("stress70b", 99, 64, 8, 128, 32, BF16, "lognormal",
                          (2048.0, 1.2, 256, 32768), 512, 64, 4, 128256),
    "prefill8": Workload("prefill8", 7, 64, 8, 128, 32, BF16, "fixed", (), 8, 0, 0, 0,
                         fixed_lens=(4096,) * 8, fixed_qlens=(1024,) * 8),
}
# Prefix sharing: the 70B batch with a 2048-token system prompt in front of every
# sequence, shared by groups of 8 consecutive sequences (their block tables point at
# the same 64 prompt pages).
WORKLOADS["shared70b"] = dataclasses.replace(WORKLOADS["stress70b"], name="shared70b",
                                             prefix_tokens=2048, prefix_group=8)
# Draft trees: the 70B batch whose 64 verify sequences each bring a random 16-node draft
# tree under the last context token (17 query tokens), attention with tree masks and
# tree verification over vocab 128256.
WORKLOADS["tree70b"] = dataclasses.replace(WORKLOADS["stress70b"], name="tree70b", k=16,
                                           tree=True)
for _base in ("stress70b", "decode64"):
    for _q in QUANTIZED:
        WORKLOADS[f"{_base}_{_q}"] = dataclasses.replace(WORKLOADS[_base], name=f"{_base}_{_q}",
                                                         kv_dtype=_q)
ORDER = ["tiny", "decode64", "verify32", "mixed272", "stress70b"]


def _rng(seed: int, stream: int) -> np.random.Generator:
    """Independent numpy stream `stream` of workload seed `seed`."""
    return np.random.default_rng([int(seed), int(stream)])


def sample_lengths(w: Workload) -> np.ndarray:
    """Context lengths L_i (KV tokens, this step's query tokens included)."""
    if w.length_law == "fixed":
        return np.asarray(w.fixed_lens, dtype=np.int64)
    rng = _rng(w.seed, 1)
    n = w.num_seqs
    if w.length_law == "lognormal":
        median, sigma, lo, hi = w.length_args
        z = rng.standard_normal(n)
        L = np.rint(np.exp(math.log(median) + sigma * z))
        return np.clip(L, lo, hi).astype(np.int64)
    if w.length_law == "uniform":
        lo, hi = w.length_args
        return rng.integers(lo, hi + 1, size=n).astype(np.int64)
    if w.length_law == "pareto":
        alpha, xmin, cap = w.length_args
        u = rng.random(n)
        L = np.floor(xmin * (1.0 - u) ** (-1.0 / alpha))
        return np.minimum(L, cap).astype(np.int64)
    raise ValueError(w.length_law)


def query_lengths(w: Workload) -> np.ndarray:
    """1 for decode sequences, k+1 for verify sequences (positions seeded-random)."""
    if w.fixed_qlens is not None:
        return np.asarray(w.fixed_qlens, dtype=np.int64)
    ql = np.ones(w.num_seqs, dtype=np.int64)
    if w.num_verify:
        idx = _rng(w.seed, 2).permutation(w.num_seqs)[: w.num_verify]
        ql[np.sort(idx)] = w.k + 1
    return ql


def build_pool(lens: np.ndarray, page_size: int, seed: int, pool_pages: Optional[int] = None,
               prefix_pages: int = 0, prefix_group: int = 0):
    """Block table [B, max_pages] (padded with -1) over a seeded random permutation of
    the pool.  With prefix_pages, consecutive groups of prefix_group sequences share
    their first prefix_pages pages (one copy per group).  Returns (block_table int32,
    num_pages)."""
    if prefix_pages:
        return _build_shared_pool(lens, page_size, seed, prefix_pages, prefix_group)
    npages = (lens + page_size - 1) // page_size
    total = int(npages.sum())
    num_pages = total if pool_pages is None else int(pool_pages)
    if num_pages < total:
        raise ValueError("pool too small for the batch")
    perm = _rng(seed, 3).permutation(num_pages)[:total]
    maxp = max(int(npages.max()) if len(npages) else 0, 1)
    bt = np.full((len(lens), maxp), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(npages):
        bt[i, :n] = perm[off:off + n]
        off += n
    return bt, num_pages


def _build_shared_pool(lens, page_size, seed, prefix_pages, group):
    npages = (lens + page_size - 1) // page_size
    if np.any(npages <= prefix_pages):
        raise ValueError("every sequence must extend past the shared prefix")
    groups = (len(lens) + group - 1) // group
    total = groups * prefix_pages + int((npages - prefix_pages).sum())
    perm = _rng(seed, 3).permutation(total)
    bt = np.full((len(lens), int(npages.max())), -1, dtype=np.int32)
    off = 0
    for gi in range(groups):
        shared = perm[off:off + prefix_pages]
        off += prefix_pages
        for i in range(gi * group, min(len(lens), (gi + 1) * group)):
            bt[i, :prefix_pages] = shared
            n = int(npages[i]) - prefix_pages
            bt[i, prefix_pages:prefix_pages + n] = perm[off:off + n]
            off += n
    return bt, total


def _torch_dtype(kv_dtype: str):
    """Storage dtype of Q (and of K/V unless they are quantised)."""
    return torch.float32 if kv_dtype == F32 else torch.bfloat16


def quantize_pool(x: torch.Tensor, kv_dtype: str):
    """Codes and scales of a float pool [num_pages, P, Hkv, D]: one scale per (page,
    slot, head), stored [num_pages, Hkv, P].  Returns (codes uint8, scales float32)."""
    qmax = 448.0 if kv_dtype == FP8 else 127.0
    n, P, H, D = x.shape
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty((n, H, P), dtype=torch.float32, device=x.device)
    step = max(1, (1 << 24) // max(1, P * H * D))
    for s in range(0, n, step):
        xs = x[s:s + step].float()
        amax = xs.abs().amax(dim=-1)                                  # [n, P, H]
        sc = torch.where(amax > 0, amax / qmax, torch.ones_like(amax))
        y = (xs / sc[..., None]).clamp(-qmax, qmax)
        if kv_dtype == FP8:
            codes[s:s + step] = y.to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            codes[s:s + step] = y.round().to(torch.int8).view(torch.uint8)
        scales[s:s + step] = sc.permute(0, 2, 1)
    return codes, scales


def normal_tensor(shape, seed: int, dtype, device="cpu") -> torch.Tensor:
    """N(0, 1) values of the given storage dtype from a torch generator seeded with
    `seed` on `device` (rounded to bf16 to nearest-even when dtype is bf16)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    numel = int(np.prod(shape))
    out = torch.empty(numel, dtype=dtype, device=dev)
    chunk = 1 << 26
    for s in range(0, numel, chunk):
        e = min(numel, s + chunk)
        out[s:e] = torch.randn(e - s, generator=g, device=dev, dtype=torch.float32).to(dtype)
    return out.view(*shape)


@dataclasses.dataclass
class AttentionInputs:
    q: torch.Tensor             # [total_q_tokens, Hq, D]
    k_pages: torch.Tensor       # [num_pages, P, Hkv, D]
    v_pages: torch.Tensor
    block_table: torch.Tensor   # int32 [B, max_pages]
    seq_lens: torch.Tensor      # int32 [B]
    query_lens: torch.Tensor    # int32 [B]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_dtype: str
    k_scale: Optional[torch.Tensor] = None  # float32 [num_pages, Hkv, P] (quantised pools)
    v_scale: Optional[torch.Tensor] = None

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def total_q_tokens(self) -> int:
        return int(self.q.shape[0])


def attention_inputs(lens, qlens, *, num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype,
                     seed, pool_pages=None, pool_device="cpu", prefix_pages=0,
                     prefix_group=0) -> AttentionInputs:
    """Paged attention inputs for explicit lengths.  The page pool (every slot, used or
    not) holds N(0,1) values drawn on `pool_device`; Q is drawn on the CPU."""
    lens = np.asarray(lens, dtype=np.int64)
    qlens = np.asarray(qlens, dtype=np.int64)
    bt, num_pages = build_pool(lens, page_size, seed, pool_pages, prefix_pages, prefix_group)
    dt = _torch_dtype(kv_dtype)
    shape = (num_pages, page_size, num_kv_heads, head_dim)
    k_scale = v_scale = None
    if kv_dtype in QUANTIZED:
        k_pages, k_scale = quantize_pool(normal_tensor(shape, seed * 4 + 1, torch.float32,
                                                       pool_device), kv_dtype)
        v_pages, v_scale = quantize_pool(normal_tensor(shape, seed * 4 + 2, torch.float32,
                                                       pool_device), kv_dtype)
    else:
        k_pages = normal_tensor(shape, seed * 4 + 1, dt, pool_device)
        v_pages = normal_tensor(shape, seed * 4 + 2, dt, pool_device)
    T = int(qlens.sum())
    q = normal_tensor((T, num_q_heads, head_dim), seed * 4 + 3, dt, "cpu")
    return AttentionInputs(q, k_pages, v_pages, torch.from_numpy(bt),
                           torch.from_numpy(lens.astype(np.int32)),
                           torch.from_numpy(qlens.astype(np.int32)), num_q_heads,
                           num_kv_heads, head_dim, page_size, kv_dtype, k_scale, v_scale)


def draft_tree_parents(qlens, seed: int, extra_roots: float = 0.0) -> np.ndarray:
    """A random draft tree per sequence: int32 [sum(qlens)], each query token's parent as
    an index among its own sequence's query tokens, -1 for a root.  Token 0 is the root
    (the last accepted token); token j > 0 hangs under a uniformly drawn earlier token (a
    random recursive tree: bushy near the root, as top-k drafting makes it), or becomes a
    root of its own with probability `extra_roots` (a forest)."""
    rng = _rng(seed, 5)
    out = []
    for ql in np.asarray(qlens, dtype=np.int64):
        par = np.full(int(ql), -1, dtype=np.int32)
        for j in range(1, int(ql)):
            par[j] = -1 if rng.random() < extra_roots else int(rng.integers(0, j))
        out.append(par)
    return np.concatenate(out) if out else np.zeros(0, dtype=np.int32)


def workload_attention(name: str, pool_device="cpu") -> AttentionInputs:
    w = WORKLOADS[name]
    return attention_inputs(sample_lengths(w) + w.prefix_tokens, query_lengths(w),
                            num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                            head_dim=w.head_dim, page_size=w.page_size, kv_dtype=w.kv_dtype,
                            seed=w.seed, pool_pages=w.pool_pages, pool_device=pool_device,
                            prefix_pages=w.prefix_tokens // w.page_size,
                            prefix_group=w.prefix_group)


@dataclasses.dataclass
class VerifyInputs:
    p: np.ndarray          # float32 [B, k+1, V] target probabilities
    q: np.ndarray          # float32 [B, k, V] draft probabilities
    draft: np.ndarray      # int32 [B, k] draft tokens, x_i ~ q_i
    seed: int              # Philox seed of the call
    parents: Optional[np.ndarray] = None  # int32 [B, k]: draft trees (node i + 1's parent)

    @property
    def B(self):
        return self.p.shape[0]

    @property
    def k(self):
        return self.p.shape[1] - 1

    @property
    def V(self):
        return self.p.shape[2]


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def verify_inputs(B: int, k: int, V: int, *, seed: int, p_logit_std: float = 3.0,
                  q_noise_std: float = 1.5) -> VerifyInputs:
    """Synthetic target/draft distributions: p = softmax(N(0, p_logit_std) logits),
    q = softmax(the same logits + N(0, q_noise_std) noise); drafts drawn from q."""
    rng = _rng(seed, 4)
    p = np.empty((B, k + 1, V), dtype=np.float32)
    q = np.empty((B, k, V), dtype=np.float32)
    draft = np.empty((B, k), dtype=np.int32)
    for b in range(B):
        logits = rng.normal(0.0, p_logit_std, size=(k + 1, V))
        p64 = _softmax_rows(logits)
        p[b] = p64
        if k:
            q64 = _softmax_rows(logits[:k] + rng.normal(0.0, q_noise_std, size=(k, V)))
            q[b] = q64
            for i in range(k):
                draft[b, i] = rng.choice(V, p=q64[i] / q64[i].sum())
    return VerifyInputs(p, q, draft, seed)


def tree_verify_inputs(parents: np.ndarray, V: int, *, seed: int, p_logit_std: float = 3.0,
                       q_noise_std: float = 1.5) -> VerifyInputs:
    """Synthetic rows for verifying draft trees: parents [B, n] (node i + 1 hangs under
    node parents[b, i], 0 the root); p [B, n+1, V] and q [B, n, V] as in verify_inputs,
    node i + 1's token drawn from q row parents[b, i] (its parent's draft distribution)."""
    B, n = parents.shape
    rng = _rng(seed, 6)
    p = np.empty((B, n + 1, V), dtype=np.float32)
    q = np.empty((B, n, V), dtype=np.float32)
    draft = np.empty((B, n), dtype=np.int32)
    for b in range(B):
        logits = rng.normal(0.0, p_logit_std, size=(n + 1, V))
        p[b] = _softmax_rows(logits)
        q64 = _softmax_rows(logits[:n] + rng.normal(0.0, q_noise_std, size=(n, V)))
        q[b] = q64
        for i in range(n):
            row = q64[parents[b, i]]
            draft[b, i] = rng.choice(V, p=row / row.sum())
    return VerifyInputs(p, q, draft, seed)


def ancestor_bits(parents: np.ndarray, qlens) -> np.ndarray:
    """The attention kernel's tree encoding: per query token a uint64 with bit a set for
    every proper ancestor a among its window's tokens (parents as in
    draft_tree_parents)."""
    masks = np.zeros(len(parents), dtype=np.uint64)
    row0 = 0
    for ql in np.asarray(qlens, dtype=np.int64):
        for j in range(int(ql)):
            m, a = 0, int(parents[row0 + j])
            while a >= 0:
                m |= 1 << a
                a = int(parents[row0 + a])
            masks[row0 + j] = m
        row0 += int(ql)
    return masks


def workload_verify(name: str, attn_parents: Optional[np.ndarray] = None) -> Optional[VerifyInputs]:
    """The workload's verification inputs.  For a tree workload, attn_parents are the
    query windows' trees (draft_tree_parents of the query lengths): each verify window's
    nodes 1..k hang where its query tokens 1..k do."""
    w = WORKLOADS[name]
    if not w.vocab:
        return None
    if w.tree:
        qlens = query_lengths(w)
        row0 = np.concatenate([[0], np.cumsum(qlens)])
        verify = [i for i in range(len(qlens)) if qlens[i] > 1]
        par = np.stack([attn_parents[row0[i] + 1:row0[i + 1]] for i in verify]).astype(np.int32)
        par = np.maximum(par, 0)
        v = tree_verify_inputs(par, w.vocab, seed=w.seed, p_logit_std=w.p_logit_std,
                               q_noise_std=w.q_noise_std)
        return dataclasses.replace(v, parents=par)
    return verify_inputs(w.num_verify, w.k, w.vocab, seed=w.seed, p_logit_std=w.p_logit_std,
                         q_noise_std=w.q_noise_std)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) of a CPU bf16 tensor, for the oracle."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def storage_for_oracle(t: torch.Tensor, kv_dtype: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return bf16_bits(t) if kv_dtype == BF16 else t.numpy()
