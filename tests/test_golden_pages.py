"""The oracle and the roofline arithmetic against numbers the pages print (CPU only).

The values live in ``golden/page_budget.txt`` with their sources.
"""
import math
import os

import numpy as np

import datagen
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def golden():
    vals = {}
    with open(os.path.join(HERE, "golden", "page_budget.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split()
                vals[key] = int(val)
    return vals


def test_oracle_attends_to_at_most_the_printed_budget():
    """Selection with the pages' (Bk, k) and q = 0 attention: lse = ln |J|, |J| <= k Bk, equal at block ends."""
    gv = golden()
    Bk, k = gv["block_size"], gv["top_k_incl_local"]
    assert Bk * k == gv["budget_tokens"]
    nb = k + 3
    N, G, d_I, d = nb * Bk, 1, 16, 8
    q_idx = datagen.host_normal(N * G * d_I, 91, 4).reshape(N, G, d_I)
    k_idx = datagen.host_normal(N * d_I, 91, 5).reshape(N, d_I)
    rows = np.array([Bk - 1, k * Bk - 2, k * Bk - 1, (k + 1) * Bk - 1, (k + 1) * Bk + 5, N - 1], np.int64)
    blk, _ = oracle.select_blocks(q_idx[rows], k_idx, rows, N, Bk, k)  # [G, rows, k]
    q = np.zeros((len(rows), 1, d), np.uint16)
    K = datagen.host_normal(N * d, 91, 2).reshape(N, 1, d)
    V = datagen.host_normal(N * d, 91, 3).reshape(N, 1, d)
    _, lse = oracle.sparse_attn(q, K, V, blk, rows, Bk, 1.0)
    count = np.exp(lse[:, 0])
    expect = [min(t + 1, (k - 1) * Bk + t % Bk + 1) for t in rows]
    np.testing.assert_allclose(count, expect, rtol=1e-12)
    assert abs(count.max() - gv["budget_tokens"]) < 1e-9
    assert np.all(count <= gv["budget_tokens"] + 1e-9)


def test_decode_roofline_bytes_follow_the_printed_cache_sizes():
    """256 B of index key per token (d_I = 128 in bf16) is ~6% of the main K/V bytes per token and layer."""
    gv = golden()
    cfg = datagen.CONFIGS["decode_1m"]
    assert cfg.d_I * 2 == gv["index_key_bytes_per_token"]
    main = gv["main_kv_heads"] * gv["main_head_dim"] * 2 * gv["main_bytes_per_element"]
    assert round(100 * gv["index_key_bytes_per_token"] / main) == gv["index_to_main_percent"]
    # the decode roofline's algorithmic bytes: the whole index-key cache plus k blocks of K and V
    per_seq = cfg.ctx * gv["index_key_bytes_per_token"] + cfg.k * cfg.Bk * 2 * cfg.H_kv * cfg.d * 2
    assert cfg.B * per_seq == 1107296256
    assert math.isclose(cfg.k * cfg.Bk, gv["budget_tokens"])
