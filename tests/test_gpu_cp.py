"""GPU parity of the context-parallel steps (kda_piece_forward,
kda_pieces_scan, kda_piece_fixup) through the C ABI: the pieces of one
sequence, run in one process and on two gloo ranks sharing this GPU (the
ranks exchange the (M, X) state pairs over gloo, through host memory; their
kernels never wait on each other), against one oracle pass over the whole
sequence."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import chunked_gated_delta_11_gb300 as kda
from chunked_gated_delta_11_gb300 import synth
from chunked_gated_delta_11_gb300.cp import LibkdaPieces
from kda_testlib import assert_close, f64, oracle_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cuts,init", [([0, 300, 477, 1000], True), ([0, 16, 16, 129], False),
                                       ([0, 2000, 4096], True)])
def test_pieces_in_one_process(cuts, init):
    kda.build.build()
    inp = synth.make_inputs(cuts[-1], 3, 1, seed=123, init_std=0.02 if init else None)
    d = {key: (t.cuda() if isinstance(t, torch.Tensor) else t) for key, t in inp.items()}
    ops = LibkdaPieces()
    outs, xs, ms, ys = [], [], [], []
    for r in range(len(cuts) - 1):
        sl = slice(cuts[r], cuts[r + 1])
        o, x, m, y = ops.piece_forward(*(d[key][sl].contiguous() for key in
                                         ("q", "k", "v", "g_raw", "beta_raw")),
                                       d["scale"], d["lower_bound"],
                                       d["initial_state"][0] if (r == 0 and init) else None,
                                       r == 0)
        outs.append(o), xs.append(x), ys.append(y)
        ms.append(torch.zeros_like(x) if m is None else m)
    s0, final = ops.scan(torch.stack(xs), torch.stack(ms))
    for r in range(1, len(outs)):
        ops.fixup(outs[r], ys[r], s0[r])
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    ro, rs = oracle_case(inp)
    assert_close(f64(torch.cat(outs)), ro, f"pieces {cuts} out")
    assert_close(f64(final)[None], rs, f"pieces {cuts} final_state")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, cuts, q):
    import torch.distributed as dist
    from chunked_gated_delta_11_gb300.cp import kda_forward_context_parallel
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        kda.load()
        inp = synth.make_inputs(cuts[-1], 4, 1, seed=321, init_std=0.02)
        sl = slice(cuts[rank], cuts[rank + 1])
        piece = [inp[key][sl].contiguous().cuda() for key in ("q", "k", "v", "g_raw", "beta_raw")]
        out, final = kda_forward_context_parallel(*piece, inp["scale"], inp["lower_bound"],
                                                  inp["initial_state"][0].cuda())
        torch.cuda.synchronize()
        # numpy arrays pickle by value: a torch tensor would go through this
        # process's file-descriptor sharer, which may be gone once it exits
        q.put((rank, kda.kda_device_status(), out.cpu().float().numpy(), final.cpu().numpy()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_on_this_gpu():
    kda.build.build()
    cuts = [0, 700, 1500]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, cuts, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in range(2)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert all(r[1] == 0 for r in res)
    inp = synth.make_inputs(cuts[-1], 4, 1, seed=321, init_std=0.02)
    ro, rs = oracle_case(inp)
    assert_close(np.concatenate([r[2] for r in res]).astype(np.float64), ro, "two ranks out")
    for r in res:
        assert_close(r[3].astype(np.float64)[None], rs, f"rank {r[0]} final_state")
