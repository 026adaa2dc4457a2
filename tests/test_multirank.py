"""The multi-rank path of the benchmark on CPU (gloo, world size 2): each
rank runs an independent replica (distinct seeds, no collective on the data
path) and the timings reduce to the maximum over ranks."""
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth
    cfg = synth.get("llama13b")
    st = synth.build(cfg.replace(seed=cfg.seed + rank), num_seqs=8)
    local = {"step_ms": 1.0 + rank, "decode_ms": 0.5 * (2 - rank)}
    agg = bench.aggregate(local, world)
    results[rank] = (agg, st.context_lens.tolist())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        r0, r1 = results[0], results[1]
    assert r0[0] == r1[0] == {"step_ms": 2.0, "decode_ms": 1.0}
    assert r0[1] != r1[1]  # replicas draw different workloads
