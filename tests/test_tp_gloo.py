"""The tensor-parallel orchestration (one shard per rank, a sum all-reduce of
the fp32 partial outputs, one bf16 rounding) with two and four gloo ranks on
the CPU.  Each rank's shard is stood in for by the oracle's partial output of
that shard (the GPU shards are checked against the same partials in
tests/test_gpu_tp.py); the reduced, rounded output must be the whole layer's
(the parity bars of every test) and the same on every rank."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as tdist
    import oracle
    import synth
    from fp8_mxfp4_expert_bf16_b300.tp import TensorParallelMoE
    tdist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    inp = synth.custom_inputs(6, 256, 4, 512, 2, seed=45)
    c = inp.cfg
    f = oracle.forward(inp.x, inp.router_w, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, c.k, c.score_func,
                       inp.logit_bias, inp.sel_bias)
    part = oracle.tp_partials(f, inp.w2_q, inp.w2_s, world)[rank]

    class OracleShard:
        """Stands in for this rank's GPU shard: its fp32 partial output."""

        def forward_partial(self, x, y32=None):
            p = torch.from_numpy(part.astype(np.float32))
            if y32 is None:
                return p
            y32.copy_(p)
            return y32

    tp = TensorParallelMoE(OracleShard(), round_bf16=lambda y32, y: y32.to(torch.bfloat16))
    y = tp.forward(torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16))
    tdist.barrier()
    tdist.destroy_process_group()
    out.put((rank, y.view(torch.int16).numpy().view(np.uint16), f.y))


@pytest.mark.parametrize("world", [2, 4])
def test_tp_allreduce_of_shard_partials_gives_the_layer(world):
    import torch.multiprocessing as mp
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from parity import check_y
    port = 29700 + world + os.getpid() % 500
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    y0 = res[0][1]
    for _, y, _ in res:
        assert np.array_equal(y, y0)                 # every rank holds the same output
    rel, mx = check_y(y0, res[0][2])                 # and it is the whole layer's
    assert rel < 1e-4
