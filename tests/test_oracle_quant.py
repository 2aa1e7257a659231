"""Pins for the oracle's quantised KV pages (CPU only).

"llm-inference-optimization-batching" (tempatgunting.com), section "Quantization and
Precision Choices for KV": INT8 or FP8 KV pages with per-head or per-token scales,
separate for K and V, dequantised inside the attention.  The oracle decodes every code
from its format's definition, multiplies by its (token, head) scale and runs the
float64 attention unchanged.  The witnesses: torch's own float8_e4m3fn decoding,
two's-complement bytes, and dense SDPA on values decoded by torch.
"""
import numpy as np
import torch

import oracle
from verify_attention_spec_gb300 import workloads as wl

from test_oracle_attention import dense_reference


def test_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8).reshape(1, 1, 1, 256)
    got = oracle.dequant_kv(codes, np.ones((1, 1, 1), np.float32), oracle.Q_E4M3).ravel()
    want = torch.from_numpy(codes.ravel()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)])
    # from the format's definition: bias 7, 3 mantissa bits, subnormals, 448, one NaN
    assert got[0x00] == 0.0 and np.signbit(got[0x80])
    assert got[0x01] == 2.0 ** -9 and got[0x07] == 7 * 2.0 ** -9
    assert got[0x08] == 2.0 ** -6 and got[0x38] == 1.0 and got[0xB8] == -1.0
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and np.isnan(got).sum() == 2


def test_int8_decode_is_twos_complement():
    codes = np.arange(256, dtype=np.uint8).reshape(1, 1, 1, 256)
    got = oracle.dequant_kv(codes, np.full((1, 1, 1), 0.5, np.float32), oracle.Q_INT8).ravel()
    np.testing.assert_array_equal(got, 0.5 * codes.ravel().view(np.int8).astype(np.float64))


def test_scale_layout_is_page_head_slot():
    """Codes all 1: every decoded element is its own scale, read at [page, head, slot]."""
    rng = np.random.default_rng(0)
    n, P, H, D = 3, 4, 2, 5
    scales = rng.random((n, H, P)).astype(np.float32) + 0.5
    got = oracle.dequant_kv(np.ones((n, P, H, D), np.uint8), scales, oracle.Q_INT8)
    for pg in range(n):
        for t in range(P):
            for h in range(H):
                assert np.all(got[pg, t, h] == np.float64(scales[pg, h, t]))


def _torch_decode(codes: torch.Tensor, scales: torch.Tensor, kv_dtype: str) -> np.ndarray:
    if kv_dtype == wl.FP8:
        x = codes.view(torch.float8_e4m3fn).to(torch.float64)
    else:
        x = codes.view(torch.int8).to(torch.float64)
    return (x * scales.permute(0, 2, 1).to(torch.float64)[..., None]).numpy()


def test_quantised_attention_against_dense_sdpa():
    """Whole path: the generator's codes and scales, decoded by torch, laid out densely
    per sequence and fed to float64 SDPA, against the oracle on the paged pool."""
    lens, qlens = [37, 5, 70, 16], [1, 3, 6, 16]
    for kv in wl.QUANTIZED:
        a = wl.attention_inputs(lens, qlens, num_q_heads=4, num_kv_heads=2, head_dim=32,
                                page_size=16, kv_dtype=kv, seed=11)
        fmt = oracle.Q_E4M3 if kv == wl.FP8 else oracle.Q_INT8
        q_bits = wl.bf16_bits(a.q)
        out, lse = oracle.paged_attn_quant(q_bits, a.k_pages.numpy(), a.v_pages.numpy(),
                                           a.k_scale.numpy(), a.v_scale.numpy(),
                                           a.block_table.numpy(), a.seq_lens.numpy(),
                                           a.query_lens.numpy(), fmt=fmt)
        kd = _torch_decode(a.k_pages, a.k_scale, kv)
        vd = _torch_decode(a.v_pages, a.v_scale, kv)
        bt = a.block_table.numpy()
        qf = a.q.to(torch.float64).numpy()
        qs, dk, dv, row = [], [], [], 0
        for i, (L, ql) in enumerate(zip(lens, qlens)):
            pos = np.arange(L)
            dk.append(kd[bt[i][pos // 16], pos % 16])
            dv.append(vd[bt[i][pos // 16], pos % 16])
            qs.append(qf[row:row + ql])
            row += ql
        ro, rl = dense_reference(qs, dk, dv, qlens, 4, 2, 1 / np.sqrt(32))
        np.testing.assert_allclose(out, ro, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse, rl, rtol=1e-10, atol=1e-12)


def test_generator_round_trip_error():
    """The input generator's codes reproduce the drawn values within half a code step:
    relative 2^-4 of the value for E4M3 (3 mantissa bits; subnormals within 2^-10 of the
    scale), and half the scale for INT8."""
    x = torch.randn(6, 16, 2, 64, generator=torch.Generator().manual_seed(3))
    for kv in wl.QUANTIZED:
        codes, scales = wl.quantize_pool(x, kv)
        back = _torch_decode(codes, scales, kv)
        err = np.abs(back - x.double().numpy())
        sc = scales.permute(0, 2, 1).double().numpy()[..., None]
        if kv == wl.FP8:
            assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(x.double().numpy()),
                                            2.0 ** -10 * sc) * (1 + 1e-6))
        else:
            assert np.all(err <= 0.5 * sc * (1 + 1e-6))
        # each (token, head) uses its full range: the largest code is the format's max
        amax = np.abs(back).max(axis=-1)
        np.testing.assert_allclose(amax, sc[..., 0] * (448.0 if kv == wl.FP8 else 127.0),
                                   rtol=1e-6)
