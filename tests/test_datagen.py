"""The seeded input generator (CPU side): determinism, statistics, row access, needle recipe."""
import math

import numpy as np

import datagen
from datagen import bf16_to_f64


def test_normal_stream_is_deterministic_and_standard():
    a = datagen.host_normal(1 << 20, 7, 1)
    b = datagen.host_normal(1 << 20, 7, 1)
    assert np.array_equal(a, b)
    c = datagen.host_normal(1 << 20, 7, 2)
    assert not np.array_equal(a, c)
    x = bf16_to_f64(a)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    assert np.abs(x).max() < 4.95
    # offsets address the same stream
    d = datagen.host_normal(1000, 7, 1, first=12345)
    assert np.array_equal(d, a[12345:13345])


def test_row_access_matches_full_tensor():
    full = datagen.host_normal(50 * 24, 9, 3).reshape(50, 24)
    rows = np.array([0, 7, 49, 3])
    part = datagen.host_normal_rows(rows, 24, 9, 3)
    assert np.array_equal(part, full[rows])


def test_q_idx_rows_match_full_generation_and_needle_alignment():
    cfg = datagen.make_config("dg", N=2048, H_q=4, H_kv=2, d=16, d_I=64, Bk=64, k=4, needles=3)
    full = datagen.prefill_host(cfg, want=("q_idx", "k_idx"))
    rows = np.array([5, 700, 2047, 1000])
    part = datagen.prefill_host(cfg, rows=rows, want=("q_idx",))
    assert np.array_equal(part["q_idx"], full["q_idx"][rows])
    nd = full["needles"]
    # needle tokens carry alpha * u; blocks are distinct per group and leave room for later rows
    toks = nd.tokens(cfg.Bk)
    assert len(set(toks.tolist())) == len(toks)
    assert nd.blocks.max() <= cfg.nb - 2
    krow = bf16_to_f64(full["k_idx"][toks[0]])
    assert abs(np.linalg.norm(krow) - nd.alpha) < 0.05 * nd.alpha
    # rows that picked exactly one needle are aligned with it at cosine ~0.9
    masks = datagen.pick_masks(cfg, nd, np.arange(cfg.N), np.arange(cfg.N), datagen.TID["pick"])
    cos = []
    for t in range(cfg.N):
        for g in range(cfg.G):
            mk = int(masks[t, g])
            if mk and (mk & (mk - 1)) == 0:
                n = mk.bit_length() - 1
                q = bf16_to_f64(full["q_idx"][t, g])
                u = nd.u[g * nd.m + n].astype(np.float64)
                cos.append(q @ u / np.linalg.norm(q))
    cos = np.array(cos)
    assert len(cos) > 100
    assert abs(np.median(cos) - 0.9) < 0.03
    # picks: about half of the eligible needles, capped at k - 1
    bits = np.array([bin(int(x)).count("1") for x in masks.reshape(-1)])
    assert bits.max() <= cfg.k - 1


def test_decode_needles_lie_before_the_local_block():
    cfg = datagen.make_config("dgd", kind="decode", B=3, ctx=4096, H_q=4, H_kv=2, d=16, d_I=32, Bk=128, k=4,
                              needles=2)
    ctx_len = np.array([4096, 300, 129])
    nd = datagen.make_needles(cfg, ctx_len)
    for b in range(cfg.B):
        loc = (ctx_len[b] - 1) // cfg.Bk
        vals = nd.blocks[b][nd.blocks[b] >= 0]
        assert np.all(vals < loc)


def test_sample_rows_includes_edges():
    r = datagen.sample_rows(131072, 512, 3, must=(0, 127, 128, 131071))
    assert len(r) == 512 and {0, 127, 128, 131071} <= set(r.tolist())
    assert np.all(np.diff(r) > 0)
