"""Context parallelism: one long sequence cut into contiguous pieces, one piece
per rank of a torch.distributed process group, joined by a scan of the
pieces' affine state maps ("You Could Have Come Up with Kimi Delta
Attention", sec. 4.1: each token step is S -> S A_t + beta_t v_t k^_t^T).

Per rank r (pieces in rank order):
  1. kda_piece_forward: rank 0 runs its piece from the sequence's initial
     state (out, X_0); every later rank runs its piece from zero (out = o^X,
     X_r) and, with v = 0, from the identity (M_r, y_t = M_t (s q^_t));
  2. the exchange, the only collective: all_gather of X_r and M_r
     (2 x H x 64 KiB per rank) in rank order;
  3. kda_pieces_scan on the gathered pairs (every rank, the same fp32 scan):
     S_0 of every piece and the final state;
  4. kda_piece_fixup: o_t += S_0 y_t over the rank's own piece.
The compute steps are an object with three methods (LibkdaPieces runs them in
libkda on the rank's GPU); the host logic is the same for any of them.  With
NCCL the gathered tensors stay on the GPU; with gloo they go through host
memory.
"""
from __future__ import annotations

import ctypes

import torch
import torch.distributed as dist

from . import HEAD_DIM, _check, _ptr, load


class LibkdaPieces:
    """The three steps in libkda (kda_piece_forward, kda_pieces_scan,
    kda_piece_fixup) on the current CUDA device and stream."""

    def __init__(self, per_head_gate: bool = False):
        self.gate = 1 if per_head_gate else 0

    def _stream(self):
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def piece_forward(self, q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state, first):
        T, H, D = q.shape
        out = torch.empty_like(q)
        x = torch.empty((H, D, D), dtype=torch.float32, device=q.device)
        m = y = ws = None
        if not first:
            m = torch.empty_like(x)
            y = torch.empty_like(q)
            ws = torch.empty(load().kda_piece_workspace_size(T, H), dtype=torch.uint8,
                             device=q.device)
        st = load().kda_piece_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                                      float(scale), float(lower_bound), _ptr(initial_state), T, H,
                                      D, _ptr(out), _ptr(x), _ptr(m), _ptr(y), self.gate,
                                      _ptr(ws), 0 if ws is None else ws.numel(), self._stream())
        _check(st, "kda_piece_forward")
        return out, x, m, y

    def scan(self, xs, ms):
        P, H, D, _ = xs.shape
        final = torch.empty((H, D, D), dtype=torch.float32, device=xs.device)
        _check(load().kda_pieces_scan(_ptr(xs), _ptr(ms), P, H, D, _ptr(final), self._stream()),
               "kda_pieces_scan")
        return xs, final

    def fixup(self, out, y, s0):
        T, H, D = out.shape
        ws = torch.empty(256, dtype=torch.uint8, device=out.device)
        _check(load().kda_piece_fixup(_ptr(out), _ptr(y), _ptr(s0), T, H, D, _ptr(ws), 256,
                                      self._stream()), "kda_piece_fixup")


def _all_gather(t, group, world):
    """Every rank's `t`, stacked in rank order, on t's device."""
    if dist.get_backend(group) == "gloo" and t.is_cuda:
        host = t.cpu()
        parts = [torch.empty_like(host) for _ in range(world)]
        dist.all_gather(parts, host, group=group)
        return torch.stack(parts).to(t.device)
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def kda_forward_context_parallel(q, k, v, g_raw, beta_raw, scale, lower_bound,
                                 initial_state=None, group=None, ops=None):
    """This rank's piece of one sequence: q, k, v, g_raw [T_r, H, 128], beta_raw
    [T_r, H] (per-channel gate; LibkdaPieces(per_head_gate=True) with g_raw
    [T_r, H] for the scalar one), pieces in rank order, any lengths (0 too).
    initial_state [H, 128, 128] fp32 is used by rank 0 only.  Returns (out of
    this piece [T_r, H, 128] bf16, the sequence's final state [H, 128, 128]
    fp32, the same on every rank)."""
    ops = LibkdaPieces() if ops is None else ops
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    first = rank == 0
    out, x, m, y = ops.piece_forward(q, k, v, g_raw, beta_raw, scale, lower_bound,
                                     initial_state if first else None, first)
    if world == 1:
        return out, x
    if m is None:  # rank 0 has no map; its slot is never read by the scan
        m = torch.zeros_like(x)
    xs = _all_gather(x, group, world)
    ms = _all_gather(m, group, world)
    s0, final = ops.scan(xs, ms)
    if not first:
        ops.fixup(out, y, s0[rank])
    return out, final


__all__ = ["LibkdaPieces", "kda_forward_context_parallel", "HEAD_DIM"]
