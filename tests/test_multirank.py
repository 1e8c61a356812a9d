"""The multi-rank path of bench.py on CPU: two gloo ranks, each with its own
seeded batch (weak scaling: the round exchanges no data between ranks).  The
whole-job figures take the slowest rank's time and the tokens and rows of
every rank, and each rank's round equals the same batch run alone."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _round_outputs(seed):
    import oracle as O
    import workloads as W

    cfg = W.tiny(seed=seed)
    ng = O.ngram_propose(cfg["hist"], cfg["hist_len"], cfg["n_min"], cfg["n_max"], cfg["L"], cfg["copy_cap"])
    return O.price_and_allocate(cfg["d"], cfg["c"], cfg["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree,
                                ng.copy_len, cfg["coef"], cfg["lam"], cfg["budget"], cfg["max_verify_len"],
                                cfg["policy"], cfg["draft_greedy"])


def _worker(rank, world, port, outdir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        pr = _round_outputs(1000 + rank)  # this rank's own batch
        tokens, rows = int(pr.verify_len.sum()), int(pr.row_off[-1])
        ms, job_tok, job_rows = bench.reduce_over_ranks(10.0 + 2.5 * rank, tokens, rows, world)
        np.savez(os.path.join(outdir, f"rank{rank}.npz"), ms=ms, job_tok=job_tok, job_rows=job_rows,
                 tokens=tokens, rows=rows, verify_len=pr.verify_len, row_off=pr.row_off)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling(orc, tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [dict(np.load(tmp_path / f"rank{r}.npz")) for r in range(world)]
    for r in range(world):
        assert float(res[r]["ms"]) == 12.5  # the slowest rank's time
        assert int(res[r]["job_tok"]) == sum(int(x["tokens"]) for x in res)
        assert int(res[r]["job_rows"]) == sum(int(x["rows"]) for x in res)
        alone = _round_outputs(1000 + r)  # the same batch in this process, no ranks
        assert np.array_equal(res[r]["verify_len"], alone.verify_len)
        assert np.array_equal(res[r]["row_off"], alone.row_off)
