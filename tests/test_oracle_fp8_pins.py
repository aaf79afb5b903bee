"""Pins of the oracle's FP8 (E4M3) index path, against things other than itself.

* decode of all 256 codes against torch's float8_e4m3fn (an independent library
  routine) and against values the OCP E4M3 format fixes in closed form;
* quantize: torch's float8_e4m3fn cast on in-range values, the round trip of
  every finite code, ties to the even code at every midpoint, saturation at 448;
* selection on E4M3 inputs equals the bf16 oracle's selection on the same values
  (every E4M3 value is exactly a bf16 value), and its block scores equal brute
  force token scores computed with numpy from torch-decoded values.
"""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def torch_decode(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def to_bf16_bits(x_f64):
    t = torch.from_numpy(np.ascontiguousarray(x_f64, np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def torch_quantize(x_bf16_bits, scale):
    x = torch.from_numpy(np.ascontiguousarray(x_bf16_bits, np.uint16).view(np.int16)).view(torch.bfloat16)
    p = x.to(torch.float32) * torch.tensor(scale, dtype=torch.float32)
    return p.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


ALL = np.arange(256, dtype=np.uint8)
NAN_CODES = {0x7F, 0xFF}


def test_decode_matches_torch_on_every_code():
    ours, ref = oracle.e4m3_decode(ALL), torch_decode(ALL)
    for c in range(256):
        if c in NAN_CODES:
            assert math.isnan(ours[c]) and math.isnan(ref[c])
        else:
            assert ours[c] == ref[c], (hex(c), ours[c], ref[c])
            assert math.copysign(1.0, ours[c]) == math.copysign(1.0, ref[c])


def test_decode_closed_forms():
    v = oracle.e4m3_decode(np.array([0x38, 0x7E, 0x01, 0x07, 0x08, 0xC0, 0x00, 0x80, 0x3F, 0x30], np.uint8))
    assert v[0] == 1.0
    assert v[1] == 448.0             # largest finite: 1.75 * 2^8
    assert v[2] == 2.0 ** -9         # smallest subnormal
    assert v[3] == 7 * 2.0 ** -9     # largest subnormal
    assert v[4] == 2.0 ** -6         # smallest normal
    assert v[5] == -2.0
    assert v[6] == 0.0 and math.copysign(1.0, v[7]) == -1.0
    assert v[8] == 1.875
    assert v[9] == 0.5
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)  # codes 0..0x7E are in increasing order


def test_quantize_round_trips_every_finite_code():
    finite = np.array([c for c in range(256) if c not in NAN_CODES], np.uint8)
    vals = oracle.e4m3_decode(finite)
    back = oracle.e4m3_quantize(to_bf16_bits(vals), 1.0)
    assert np.array_equal(back, finite)


def test_quantize_ties_to_even_at_midpoints():
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        mid = (lo + hi) / 2  # needs 4 significant bits: exact in bf16
        bits = to_bf16_bits(np.array([mid]))
        assert float(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double()) == mid
        even = c if (c & 1) == 0 else c + 1
        assert oracle.e4m3_quantize(bits, 1.0)[0] == even, hex(c)
        # one bf16 step either side of the midpoint rounds to the nearer code
        above = np.array([bits[0] + 1], np.uint16)
        below = np.array([bits[0] - 1], np.uint16)
        if mid > 0:
            assert oracle.e4m3_quantize(above, 1.0)[0] == c + 1
            assert oracle.e4m3_quantize(below, 1.0)[0] == c
        neg = np.array([bits[0] | 0x8000], np.uint16)
        assert oracle.e4m3_quantize(neg, 1.0)[0] == (even | 0x80)


def test_quantize_saturates_at_448():
    x = to_bf16_bits(np.array([448.0, 460.0, 464.0, 500.0, 1e6, -1e30, 3e38, -449.0]))
    assert oracle.e4m3_quantize(x, 1.0).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]
    # the scale is applied before rounding: 100 * 8 = 800 -> 448
    assert oracle.e4m3_quantize(to_bf16_bits(np.array([100.0])), 8.0)[0] == 0x7E


@pytest.mark.parametrize("scale", [1.0, 0.37, 16.0])
def test_quantize_matches_torch_in_range(scale):
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000) * 30.0, rng.standard_normal(5000) * 1e-2,
                        rng.standard_normal(2000) * 1e-4])
    x = x[np.abs(x * scale) < 440.0]
    bits = to_bf16_bits(x)
    assert np.array_equal(oracle.e4m3_quantize(bits, scale), torch_quantize(bits, scale))


def _random_codes(rng, shape, spread=2.0):
    """E4M3 codes of seeded normal values (through torch's cast, never the oracle's)."""
    x = rng.standard_normal(shape) * spread
    return torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("N,G,d_I,Bk,k", [(700, 2, 64, 64, 5), (1100, 1, 128, 128, 4), (512, 3, 32, 64, 3)])
def test_select_e4m3_equals_bf16_select_on_the_same_values(N, G, d_I, Bk, k):
    rng = np.random.default_rng(N + G)
    q8, k8 = _random_codes(rng, (N, G, d_I)), _random_codes(rng, (N, d_I))
    qb, kb = to_bf16_bits(torch_decode(q8)), to_bf16_bits(torch_decode(k8))
    rows = np.arange(N)
    b8, kth8 = oracle.select_blocks_e4m3(q8, k8, rows, N, Bk, k)
    b16, kth16 = oracle.select_blocks(qb, kb, rows, N, Bk, k)
    assert np.array_equal(b8, b16)
    assert np.array_equal(kth8, kth16)
    S8 = oracle.block_scores_e4m3(q8, k8, rows, N, Bk)
    S16 = oracle.block_scores(qb, kb, rows, N, Bk)
    assert np.array_equal(S8, S16)


def test_block_scores_e4m3_brute_force():
    N, G, d_I, Bk = 300, 2, 64, 64
    rng = np.random.default_rng(3)
    q8, k8 = _random_codes(rng, (N, G, d_I)), _random_codes(rng, (N, d_I))
    qf, kf = torch_decode(q8), torch_decode(k8)
    s = np.einsum("tgc,jc->tgj", qf, kf) / math.sqrt(d_I)  # token scores, every pair
    nb = (N + Bk - 1) // Bk
    ref = np.full((N, G, nb), -np.inf)
    for t in range(N):
        for b in range(t // Bk + 1):
            ref[t, :, b] = s[t, :, b * Bk:min(t + 1, (b + 1) * Bk)].max(axis=1)
    S = oracle.block_scores_e4m3(q8, k8, np.arange(N), N, Bk)
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(np.isneginf(S), np.isneginf(ref))


def test_needle_inputs_fit_e4m3_range():
    """The seeded index inputs (needle keys of length 4 sqrt(d_I)) stay inside +-448, so the cast of the
    test inputs never saturates."""
    cfg = datagen.make_config("fp8_range", N=2048, H_q=8, H_kv=4, d=64, d_I=128, Bk=128, k=8, needles=4)
    inp = datagen.prefill_host(cfg, want=("q_idx", "k_idx"))
    for name in ("q_idx", "k_idx"):
        v = datagen.bf16_to_f64(inp[name])
        assert np.abs(v).max() < 448.0
