"""msa_decode_noalloc: the decode step for callers that may not allocate device memory.

Some hosts cannot let this library call cudaMalloc: a plugin whose application
owns all GPU memory, or a serving loop where an allocation could block and
synchronize the device.  msa_decode_noalloc takes its scratch from a fixed
device array inside the library instead of a workspace.  These tests call it
through the C ABI and check each result against msa_decode on the same inputs,
with the tolerance the parity tests use: two calls in a row, a larger batch
followed by a smaller one (the shared array keeps the larger call's contents),
and the largest batch whose scratch still fits the array.  The file is named so
that pytest collects it last.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

LIMIT = 8 << 20  # bytes of the fixed scratch array, as include/msa.h states


def dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


class _Inputs:
    """One decode step's device inputs and msa_decode's results on them."""

    def __init__(self, msa, cfg, ctx_len):
        import datagen
        self.cfg = cfg
        h = datagen.decode_host(cfg, np.asarray(ctx_len, np.int64))
        self.q_t, self.q_idx_t = dev_bf16(h["q_t"]), dev_bf16(h["q_idx_t"])
        self.k_idx_cache, self.k_cache = dev_bf16(h["k_idx_cache"]), dev_bf16(h["k_cache"])
        self.v_cache = dev_bf16(h["v_cache"])
        self.lens = torch.from_numpy(np.asarray(ctx_len, np.int32)).cuda()
        self.shp = msa.shape(cfg.ctx, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_I, cfg.Bk, cfg.k)
        self.scale = 1.0 / math.sqrt(cfg.d)
        ws = torch.empty(msa.msa_decode_workspace(cfg.B, self.shp), dtype=torch.uint8, device="cuda")
        out, lse, blk = self._outputs()
        msa.msa_decode(self.q_t, self.q_idx_t, self.k_idx_cache, self.k_cache, self.v_cache, self.lens, cfg.B,
                       self.shp, self.scale, out, lse, blk, ws)
        assert msa.msa_check_device_error(ws) == 0
        self.ref = (out.float().cpu().numpy(), lse.cpu().numpy(), blk.cpu().numpy())

    def _outputs(self):
        c = self.cfg
        return (torch.full((c.B, c.H_q, c.d), float("nan"), dtype=torch.bfloat16, device="cuda"),
                torch.full((c.B, c.H_q), float("nan"), dtype=torch.float32, device="cuda"),
                torch.full((c.B, c.H_kv, c.k), -7, dtype=torch.int32, device="cuda"))

    def noalloc(self, msa, B=None):
        out, lse, blk = self._outputs()
        status = msa.raw().msa_decode_noalloc(msa._ptr(self.q_t), msa._ptr(self.q_idx_t), msa._ptr(self.k_idx_cache),
                                              msa._ptr(self.k_cache), msa._ptr(self.v_cache), msa._ptr(self.lens),
                                              self.cfg.B if B is None else B, msa.ctypes.byref(self.shp), self.scale,
                                              msa._ptr(out), msa._ptr(lse), msa._ptr(blk), msa._stream(None))
        torch.cuda.synchronize()
        return status, out, lse, blk

    def check(self, msa, what):
        status, out, lse, blk = self.noalloc(msa)
        assert status == msa.MSA_OK, (what, msa.msa_status_string(status))
        r_out, r_lse, r_blk = self.ref
        np.testing.assert_array_equal(blk.cpu().numpy(), r_blk, err_msg=what)
        o = out.float().cpu().numpy()
        assert np.all(np.abs(o - r_out) <= 2e-2 + 1e-2 * np.abs(r_out)), "%s: out differs" % what
        assert np.all(np.abs(lse.cpu().numpy() - r_lse) <= 2e-2 + 1e-2 * np.abs(r_lse)), "%s: lse differs" % what


def _cfg(name, index, **kw):
    import datagen
    return datagen.make_config(name, kind="decode", index=index, **kw)


def test_decode_noalloc_matches_decode_twice():
    from block_sparse_long_index_gb300 import msa
    cfg = _cfg("noalloc", 300, B=3, ctx=9000, H_q=16, H_kv=4, d=128, d_I=128, Bk=128, k=8, needles=2)
    inp = _Inputs(msa, cfg, [9000, 4321, 200])
    for call in range(2):
        inp.check(msa, "call %d" % call)


def test_decode_noalloc_smaller_call_after_larger_one():
    """The shared array still holds a larger call's tickets, candidate lists and partials when a smaller call
    starts; the smaller call must clear or overwrite everything it reads."""
    from block_sparse_long_index_gb300 import msa
    big = _Inputs(msa, _cfg("noalloc_big", 301, B=6, ctx=6000, H_q=32, H_kv=8, d=128, d_I=128, Bk=64, k=16,
                            needles=3), [6000, 5999, 4096, 3000, 1500, 65])
    small = _Inputs(msa, _cfg("noalloc_small", 302, B=2, ctx=4000, H_q=16, H_kv=4, d=64, d_I=64, Bk=64, k=6,
                              needles=2), [4000, 777])
    big.check(msa, "larger call")
    small.check(msa, "smaller call after the larger one")
    big.check(msa, "larger call again")


def test_decode_noalloc_at_the_edge_of_its_fixed_scratch():
    """The largest batch whose scratch (msa_decode_workspace) fits the fixed array runs and matches msa_decode;
    one more sequence is rejected with MSA_ERR_WORKSPACE_TOO_SMALL before any launch."""
    from block_sparse_long_index_gb300 import msa
    kw = dict(ctx=1024, H_q=64, H_kv=8, d=128, d_I=128, Bk=128, k=32, needles=2)
    shp = msa.shape(kw["ctx"], kw["H_q"], kw["H_kv"], kw["d"], kw["d_I"], kw["Bk"], kw["k"])
    sizes = {B: msa.msa_decode_workspace(B, shp) for B in range(1, 33)}
    b_max = max(B for B, s in sizes.items() if s <= LIMIT)
    assert b_max < 32 and sizes[b_max + 1] > LIMIT
    rng = np.random.default_rng(5)
    lens = [1024] + rng.integers(1, 1025, b_max).tolist()
    inp = _Inputs(msa, _cfg("noalloc_edge", 303, B=b_max + 1, **kw), lens)
    # the first b_max sequences of the same buffers: a batch exactly at the edge
    edge = _Inputs.__new__(_Inputs)
    edge.__dict__.update(inp.__dict__)
    edge.cfg = _cfg("noalloc_edge", 303, B=b_max, **kw)
    ws = torch.empty(sizes[b_max], dtype=torch.uint8, device="cuda")
    out, lse, blk = edge._outputs()
    msa.msa_decode(inp.q_t, inp.q_idx_t, inp.k_idx_cache, inp.k_cache, inp.v_cache, inp.lens, b_max, inp.shp,
                   inp.scale, out, lse, blk, ws)
    assert msa.msa_check_device_error(ws) == 0
    edge.ref = (out.float().cpu().numpy(), lse.cpu().numpy(), blk.cpu().numpy())
    edge.check(msa, "batch at the edge")
    status, _, _, _ = inp.noalloc(msa, B=b_max + 1)
    assert status == msa.MSA_ERR_WORKSPACE_TOO_SMALL


def test_decode_noalloc_rejects_shapes_beyond_its_fixed_scratch():
    from block_sparse_long_index_gb300 import msa
    shp = msa.shape(1 << 20, 64, 8, 128, 128, 128, 32)
    big_b = 64  # needs far more than the fixed 8 MiB of scratch
    assert msa.msa_decode_workspace(big_b, shp) > LIMIT
    fake = msa.ctypes.c_void_p(1 << 20)
    status = msa.raw().msa_decode_noalloc(fake, fake, fake, fake, fake, fake, big_b, msa.ctypes.byref(shp), 0.1,
                                          fake, None, None, None)
    assert status == msa.MSA_ERR_WORKSPACE_TOO_SMALL
