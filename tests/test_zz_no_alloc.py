"""msa_decode_noalloc: the decode step for callers that may not allocate device memory.

Some hosts cannot let this library call cudaMalloc: a plugin whose application
owns all GPU memory, or a serving loop where an allocation could block and
synchronize the device.  msa_decode_noalloc takes its scratch from a fixed
device array inside the library instead of a workspace.  This test calls it
through the C ABI twice in a row and checks each result against msa_decode on
the same inputs, with the tolerance the parity tests use.  The file is named so
that pytest collects it last.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def test_decode_noalloc_matches_decode_twice():
    import datagen
    from block_sparse_long_index_gb300 import msa

    cfg = datagen.make_config("noalloc", kind="decode", B=3, ctx=9000, H_q=16, H_kv=4, d=128, d_I=128, Bk=128,
                              k=8, needles=2)
    ctx_len = np.array([9000, 4321, 200], np.int64)
    h = datagen.decode_host(cfg, ctx_len)
    q_t, q_idx_t = dev_bf16(h["q_t"]), dev_bf16(h["q_idx_t"])
    k_idx_cache, k_cache, v_cache = dev_bf16(h["k_idx_cache"]), dev_bf16(h["k_cache"]), dev_bf16(h["v_cache"])
    lens = torch.from_numpy(ctx_len.astype(np.int32)).cuda()
    shp = msa.shape(cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
    scale = 1.0 / math.sqrt(cfg.d)

    # the existing entry point, with a caller-owned workspace
    ws = torch.empty(msa.msa_decode_workspace(cfg.B, shp), dtype=torch.uint8, device="cuda")
    ref_out = torch.empty((cfg.B, cfg.H_q, cfg.d), dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty((cfg.B, cfg.H_q), dtype=torch.float32, device="cuda")
    ref_blk = torch.empty((cfg.B, cfg.H_kv, cfg.k), dtype=torch.int32, device="cuda")
    msa.msa_decode(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, lens, cfg.B, shp, scale, ref_out, ref_lse, ref_blk, ws)
    assert msa.msa_check_device_error(ws) == 0
    r_out = ref_out.float().cpu().numpy()
    r_lse = ref_lse.cpu().numpy()

    for call in range(2):
        out = torch.full((cfg.B, cfg.H_q, cfg.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((cfg.B, cfg.H_q), float("nan"), dtype=torch.float32, device="cuda")
        blk = torch.full((cfg.B, cfg.H_kv, cfg.k), -7, dtype=torch.int32, device="cuda")
        status = msa.raw().msa_decode_noalloc(msa._ptr(q_t), msa._ptr(q_idx_t), msa._ptr(k_idx_cache),
                                              msa._ptr(k_cache), msa._ptr(v_cache), msa._ptr(lens), cfg.B,
                                              msa.ctypes.byref(shp), scale, msa._ptr(out), msa._ptr(lse),
                                              msa._ptr(blk), msa._stream(None))
        assert status == msa.MSA_OK, msa.msa_status_string(status)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(blk.cpu().numpy(), ref_blk.cpu().numpy())
        o = out.float().cpu().numpy()
        assert np.all(np.abs(o - r_out) <= 2e-2 + 1e-2 * np.abs(r_out)), "call %d: out differs" % call
        assert np.all(np.abs(lse.cpu().numpy() - r_lse) <= 2e-2 + 1e-2 * np.abs(r_lse)), "call %d: lse" % call


def test_decode_noalloc_rejects_shapes_beyond_its_fixed_scratch():
    from block_sparse_long_index_gb300 import msa
    shp = msa.shape(1 << 20, 64, 8, 128, 128, 128, 32)
    big_b = 64  # needs far more than the fixed 8 MiB of scratch
    assert msa.msa_decode_workspace(big_b, shp) > (8 << 20)
    fake = msa.ctypes.c_void_p(1 << 20)
    status = msa.raw().msa_decode_noalloc(fake, fake, fake, fake, fake, fake, big_b, msa.ctypes.byref(shp), 0.1,
                                          fake, None, None, None)
    assert status == msa.MSA_ERR_WORKSPACE_TOO_SMALL
