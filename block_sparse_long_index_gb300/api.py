"""Tensor-level entry points over the C ABI (allocation of outputs and workspaces with torch).

``MsaPrefill`` / ``MsaDecode`` own their outputs and workspace so repeated steps
allocate nothing; ``prefill`` / ``decode`` are one-shot conveniences.  All
compute is in libmsa.so.
"""
from __future__ import annotations

import math

import torch

from . import msa as _c


def _check_bf16(name, t, shape):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA bfloat16 tensor" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


class MsaPrefill:
    """One prefill layer step: select -> (invert + KV-outer attention + combine).

    Calling the object runs msa_prefill (both stages in one call); ``select``
    and ``attend`` run the two stages as separate calls."""

    def __init__(self, N, H_q, H_kv, d, d_I, Bk, k, device="cuda"):
        self.N, self.H_q, self.H_kv, self.d, self.d_I, self.Bk, self.k = N, H_q, H_kv, d, d_I, Bk, k
        self.G = H_kv
        self.shape = _c.shape(N, H_q, H_kv, d, d_I, Bk, k)
        ws = max(_c.msa_select_blocks_workspace(N, self.G, d_I, Bk, k), _c.msa_sparse_attn_fwd_workspace(self.shape),
                 _c.msa_prefill_workspace(self.shape))
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)
        self.block_idx = torch.empty((self.G, N, k), dtype=torch.int32, device=device)
        self.out = torch.empty((N, H_q, d), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((H_q, N), dtype=torch.float32, device=device)

    def select(self, q_idx, k_idx, stream=None):
        _c.msa_select_blocks(q_idx, k_idx, self.N, self.G, self.d_I, self.Bk, self.k, self.block_idx,
                             self.workspace, stream=stream)
        return self.block_idx

    def attend(self, q, k, v, block_idx=None, scale=None, stream=None, out=None, lse=None):
        """The attention stage; out / lse default to the object's own buffers."""
        scale = 1.0 / math.sqrt(self.d) if scale is None else scale
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        _c.msa_sparse_attn_fwd(q, k, v, self.block_idx if block_idx is None else block_idx, self.shape, scale,
                               out, lse, self.workspace, stream=stream)
        return out, lse

    def __call__(self, q, k, v, q_idx, k_idx, scale=None, stream=None):
        N, G = self.N, self.G
        _check_bf16("q", q, (N, self.H_q, self.d))
        _check_bf16("k", k, (N, self.H_kv, self.d))
        _check_bf16("v", v, (N, self.H_kv, self.d))
        _check_bf16("q_idx", q_idx, (N, G, self.d_I))
        _check_bf16("k_idx", k_idx, (N, self.d_I))
        scale = 1.0 / math.sqrt(self.d) if scale is None else scale
        _c.msa_prefill(q, k, v, q_idx, k_idx, self.shape, scale, self.block_idx, self.out, self.lse, self.workspace,
                       stream=stream)
        return self.out, self.lse, self.block_idx

    def device_status(self, stream=None):
        return _c.msa_check_device_error(self.workspace, stream)


class MsaDecode:
    """One decode step for B sequences over caches of capacity ctx_max."""

    def __init__(self, B, ctx_max, H_q, H_kv, d, d_I, Bk, k, device="cuda"):
        self.B, self.ctx_max = B, ctx_max
        self.H_q, self.H_kv, self.d, self.d_I, self.Bk, self.k = H_q, H_kv, d, d_I, Bk, k
        self.shape = _c.shape(ctx_max, H_q, H_kv, d, d_I, Bk, k)
        self.workspace = torch.empty(_c.msa_decode_workspace(B, self.shape), dtype=torch.uint8, device=device)
        self.out = torch.empty((B, H_q, d), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((B, H_q), dtype=torch.float32, device=device)
        self.block_idx = torch.empty((B, H_kv, k), dtype=torch.int32, device=device)

    def __call__(self, q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, scale=None, stream=None):
        scale = 1.0 / math.sqrt(self.d) if scale is None else scale
        _c.msa_decode(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, self.B, self.shape, scale, self.out,
                      self.lse, self.block_idx, self.workspace, stream=stream)
        return self.out, self.lse, self.block_idx

    def device_status(self, stream=None):
        return _c.msa_check_device_error(self.workspace, stream)


def prefill(q, k, v, q_idx, k_idx, Bk=128, k_blocks=16, scale=None):
    """One-shot prefill: returns (out [N,H_q,d] bf16, lse [H_q,N] fp32, block_idx [G,N,k] int32)."""
    N, H_q, d = q.shape
    H_kv = k.shape[1]
    run = MsaPrefill(N, H_q, H_kv, d, q_idx.shape[2], Bk, k_blocks, device=q.device)
    out, lse, blk = run(q, k, v, q_idx, k_idx, scale)
    return out, lse, blk


def decode(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, Bk=128, k_blocks=16, scale=None):
    """One-shot decode step: returns (out [B,H_q,d], lse [B,H_q], block_idx [B,G,k])."""
    B, H_q, d = q_t.shape
    _, ctx_max, H_kv, _ = k_cache.shape
    run = MsaDecode(B, ctx_max, H_q, H_kv, d, q_idx_t.shape[2], Bk, k_blocks, device=q_t.device)
    return run(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, scale)


def varlen_cells(lengths, Bk):
    """Block-aligned cell offsets for sequences of the given lengths: cu_seqlens [S+1] (a list of ints)
    for msa_select_blocks_varlen / msa_prefill_varlen, sequence s starting at the first block boundary
    after sequence s-1's last token; N = cu_seqlens[-1] cells hold them all."""
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + (int(n) + Bk - 1) // Bk * Bk)
    return cu


def prefill_from_host(run: MsaPrefill, host_inputs, dev_inputs, host_out, stream=None):
    """End-to-end step through the public API with host buffers: pinned host -> device copies,
    the prefill step, device -> pinned host copies of out and lse, all on one stream."""
    for name in ("q", "k", "v", "q_idx", "k_idx"):
        dev_inputs[name].copy_(host_inputs[name], non_blocking=True)
    out, lse, blk = run(dev_inputs["q"], dev_inputs["k"], dev_inputs["v"], dev_inputs["q_idx"], dev_inputs["k_idx"],
                        stream=stream)
    host_out["out"].copy_(out, non_blocking=True)
    host_out["lse"].copy_(lse, non_blocking=True)
    return host_out


class PrefillHostPipeline:
    """Prefill steps from pinned host buffers to pinned host buffers, with the copies overlapped.

    Copies run on two host->device and two device->host streams (each direction
    then keeps two copy engines busy, which on this GPU's host link roughly
    doubles what one stream moves while the other direction is busy too), and
    the prefill on the compute stream.  Step i's inputs land in one of two
    device input sets while step i-1 computes on the other; its index inputs
    (q_idx, k_idx) are copied first so that the select can start while q, k and
    v are still in flight.  Step i's out and lse go to one of two device output
    sets and are copied back while step i+1 computes into the other, so the
    compute stream never waits for a device->host copy of the step before.
    Every step still copies all of its inputs in and all of its outputs (out,
    lse) out."""

    NAMES = ("q_idx", "k_idx", "q", "k", "v")

    def __init__(self, run: MsaPrefill, device="cuda"):
        self.run = run
        self.dev = [{n: torch.empty(_input_shape(run, n), dtype=torch.bfloat16, device=device) for n in self.NAMES}
                    for _ in range(2)]
        self.outs = [(run.out, run.lse), (torch.empty_like(run.out), torch.empty_like(run.lse))]
        self.h2d = [torch.cuda.Stream(device=device) for _ in range(2)]
        self.d2h = [torch.cuda.Stream(device=device) for _ in range(2)]

    def __call__(self, host_inputs, host_outputs, stream=None):
        """host_inputs: list of dicts of pinned bf16 tensors (q, k, v, q_idx, k_idx), one per step;
        host_outputs: list of dicts of pinned tensors (out, lse), one per step.  Returns once the
        work is queued; it is ordered before later work on `stream` (default: the current stream)."""
        comp = torch.cuda.current_stream() if stream is None else stream
        E = torch.cuda.Event
        for st in self.h2d + self.d2h:
            st.wait_stream(comp)
        half = self.run.N // 2
        attn_done, d2h_done = {}, {}
        for i, (hin, hout) in enumerate(zip(host_inputs, host_outputs)):
            dev = self.dev[i % 2]
            idx_in, qkv_in = E(), [E(), E()]
            for j, st in enumerate(self.h2d):
                with torch.cuda.stream(st):
                    if i - 2 in attn_done:  # the attention of step i-2 has finished reading this input set
                        st.wait_event(attn_done[i - 2])
                    if j == 0:
                        for n in ("q_idx", "k_idx"):
                            dev[n].copy_(hin[n], non_blocking=True)
                        idx_in.record(st)
                        dev["q"][:half].copy_(hin["q"][:half], non_blocking=True)
                        dev["k"].copy_(hin["k"], non_blocking=True)
                    else:
                        dev["q"][half:].copy_(hin["q"][half:], non_blocking=True)
                        dev["v"].copy_(hin["v"], non_blocking=True)
                    qkv_in[j].record(st)
            comp.wait_event(idx_in)
            self.run.select(dev["q_idx"], dev["k_idx"], stream=comp)
            for ev in qkv_in:
                comp.wait_event(ev)
            for ev in d2h_done.get(i - 2, ()):  # out and lse of step i-2 (this output set) are on the host
                comp.wait_event(ev)
            out, lse = self.outs[i % 2]
            self.run.attend(dev["q"], dev["k"], dev["v"], stream=comp, out=out, lse=lse)
            attn_done[i] = E()
            attn_done[i].record(comp)
            d2h_done[i] = []
            for j, st in enumerate(self.d2h):
                with torch.cuda.stream(st):
                    st.wait_event(attn_done[i])
                    if j == 0:
                        hout["out"][:half].copy_(out[:half], non_blocking=True)
                        hout["lse"].copy_(lse, non_blocking=True)
                    else:
                        hout["out"][half:].copy_(out[half:], non_blocking=True)
                    ev = E()
                    ev.record(st)
                    d2h_done[i].append(ev)
        for st in self.h2d + self.d2h:
            comp.wait_stream(st)
        return host_outputs


def _input_shape(run: MsaPrefill, name):
    return {"q": (run.N, run.H_q, run.d), "k": (run.N, run.H_kv, run.d), "v": (run.N, run.H_kv, run.d),
            "q_idx": (run.N, run.G, run.d_I), "k_idx": (run.N, run.d_I)}[name]
