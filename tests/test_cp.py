"""The host logic of the context-parallel split (chunked_gated_delta_11_gb300/cp.py)
on CPU gloo ranks: the pieces of one sequence on 2 and 3 ranks, the exchange
of the (M, X) state pairs, the scan and the fix-up, with the three compute
steps done by the fp64 oracle (X from zero or the initial state; M and y from
the identity with v = 0).  The joined result must equal one oracle pass over
the whole sequence to fp64 rounding: the split is exact ("You Could Have Come
Up with Kimi Delta Attention", sec. 4.1)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from chunked_gated_delta_11_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OraclePieces:
    """The three steps of cp.py in fp64 by the oracle (tests only)."""

    def piece_forward(self, q, k, v, g, beta, scale, lb, init, first):
        import oracle
        f = lambda t: t.double().numpy()
        T, H, D = q.shape
        init_np = None if init is None else init.double().numpy()[None]
        out, x = oracle.fwd_raw(f(q), f(k), f(v), f(g), f(beta), scale, lb, init_np)
        if first:
            return torch.from_numpy(out), torch.from_numpy(x[0]), None, None
        eye = np.broadcast_to(np.eye(D), (1, H, D, D)).copy()
        y, m = oracle.fwd_raw(f(q), f(k), np.zeros((T, H, D)), f(g), f(beta), scale, lb, eye)
        return (torch.from_numpy(out), torch.from_numpy(x[0]), torch.from_numpy(m[0]),
                torch.from_numpy(y))

    def scan(self, xs, ms):
        xs = xs.clone()
        S = xs[0].clone()
        for j in range(1, xs.shape[0]):
            nxt = S @ ms[j] + xs[j]
            xs[j] = S
            S = nxt
        return xs, S

    def fixup(self, out, y, s0):
        out += torch.einsum("hvk,thk->thv", s0, y)


def _worker(rank, world, port, cuts, q):
    import torch.distributed as dist
    from chunked_gated_delta_11_gb300.cp import kda_forward_context_parallel
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = synth.make_inputs(cuts[-1], 2, 1, seed=77, init_std=0.02)
        sl = slice(cuts[rank], cuts[rank + 1])
        piece = [inp[key][sl] for key in ("q", "k", "v", "g_raw", "beta_raw")]
        out, final = kda_forward_context_parallel(*piece, inp["scale"], inp["lower_bound"],
                                                  inp["initial_state"][0], ops=OraclePieces())
        q.put((rank, out.numpy(), final.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [[0, 40, 97], [0, 33, 33, 150]])
def test_context_parallel_split_is_exact_on_cpu_ranks(cuts):
    import oracle
    world = len(cuts) - 1
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cuts, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    inp = synth.make_inputs(cuts[-1], 2, 1, seed=77, init_std=0.02)
    f = lambda t: t.double().numpy()
    ro, rs = oracle.fwd_raw(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["g_raw"]),
                            f(inp["beta_raw"]), inp["scale"], inp["lower_bound"],
                            f(inp["initial_state"]))
    out = np.concatenate([r[1] for r in res])
    assert np.abs(out - ro).max() <= 1e-10 * np.abs(ro).max()
    for r in res:  # every rank holds the final state
        assert np.abs(r[2] - rs[0]).max() <= 1e-10 * np.abs(rs).max()
