"""Warmup mode on the GPU against the oracle: dense causal attention (out, lse), the index branch's lse, and
the KL of every row with its gradients on q^I and k^I ("MSA" study note 4-4)."""
import math

import numpy as np
import pytest
import torch

import datagen
import oracle
from parity import bf16_tensor_to_f64, compare_attn
from test_gpu_bwd import rel_report

pytestmark = pytest.mark.gpu

CASES = [
    # name, N, H_q, H_kv, d, d_I
    ("tiny_one_tile", 16, 4, 1, 64, 32),
    ("single_row", 1, 2, 2, 64, 64),
    ("ragged_gs4", 300, 8, 2, 64, 32),
    ("gs8_d128", 1000, 16, 2, 128, 128),
    ("gs1_dI64", 777, 4, 4, 128, 64),
    ("gs2_long", 2100, 8, 4, 128, 128),
    # the tensor-core path (d = d_I = 128, gs = 8): one key tile exactly, a partial tile, ragged with 3 groups
    ("tc_one_key_tile", 128, 8, 1, 128, 128),
    ("tc_partial_tile", 17, 8, 1, 128, 128),
    ("tc_ragged_g3", 3001, 24, 3, 128, 128),
]


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def run_warmup(msa, h, N, H_q, H_kv, d, d_I, scale, w):
    G = H_kv
    shp = msa.shape(N, H_q, H_kv, d, d_I, 64, 1)
    q, k, v, qi, ki = dev(h["q"]), dev(h["k"]), dev(h["v"]), dev(h["q_idx"]), dev(h["k_idx"])
    out = torch.full((N, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H_q, N), float("nan"), dtype=torch.float32, device="cuda")
    lse_idx = torch.full((G, N), float("nan"), dtype=torch.float32, device="cuda")
    msa.msa_warmup_fwd(q, k, v, qi, ki, shp, scale, out, lse, lse_idx)
    dq_idx = torch.full((N, G, d_I), float("nan"), dtype=torch.float32, device="cuda")
    dk_idx = torch.full((N, d_I), float("nan"), dtype=torch.float32, device="cuda")
    kl = torch.full((G, N), float("nan"), dtype=torch.float32, device="cuda")
    msa.msa_warmup_index_grad(q, k, qi, ki, lse, lse_idx, shp, scale, w, dq_idx, dk_idx, kl)
    torch.cuda.synchronize()
    return out, lse, lse_idx, dq_idx, dk_idx, kl


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_warmup_parity(case):
    from block_sparse_long_index_gb300 import msa
    name, N, H_q, H_kv, d, d_I = case
    cfg = datagen.make_config("wu_" + name, N=N, H_q=H_q, H_kv=H_kv, d=d, d_I=d_I, Bk=64, k=1, needles=0)
    h = datagen.prefill_host(cfg)
    scale, w = 1.0 / math.sqrt(d), 0.7
    out, lse, lse_idx, dq_idx, dk_idx, kl = run_warmup(msa, h, N, H_q, H_kv, d, d_I, scale, w)
    rows = np.arange(N)
    ref_o, ref_l = oracle.dense_attn(h["q"], h["k"], h["v"], rows, scale)
    rep = compare_attn(bf16_tensor_to_f64(out), lse.T.cpu().numpy().astype(np.float64), ref_o, ref_l)
    ref = oracle.warmup_index(h["q"], h["k"], h["q_idx"], h["k_idx"], scale, w)
    lerr = np.abs(lse_idx.cpu().numpy() - ref["lse_idx"])
    assert float(lerr.max()) <= 2e-2 + 1e-2 * float(np.abs(ref["lse_idx"]).max()), float(lerr.max())
    reps = {}
    for nm, gpu in (("kl", kl), ("dq_idx", dq_idx), ("dk_idx", dk_idx)):
        g = gpu.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all(), nm
        if np.abs(ref[nm]).max() == 0.0:  # one key per row: nothing to learn
            assert np.abs(g).max() <= 1e-6, nm
            continue
        reps[nm] = rel_report(g, ref[nm])
    print(name, rep, reps)
    for nm, r in reps.items():
        assert r["ok"], (nm, r)
