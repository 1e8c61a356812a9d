"""Two processes on one GPU, each with its own workspace and batch: every
launch of one process's rounds must give that process's oracle results while
the other process's rounds run on the same device (separate contexts, no
shared device state, no kernel that waits on another launch).  The processes
step together through gloo barriers, so their launches overlap in time."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

RATES = (0.30, 0.60)  # each process's batch: the editing workload at its own edit rate
STEPS = 6


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _child(rank, world, port, outdir):
    import datetime

    import torch
    import torch.distributed as dist

    import oracle as O
    import speculative_decoding_draft_spec_gb300 as S
    import workloads as W
    from speculative_decoding_draft_spec_gb300.round import ChainRound

    from ._gpu import compare_sampled, gpu_chain, logits_dev

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=300))
    torch.cuda.set_device(0)
    checked = 0
    try:
        S.load()
        # greedy: the whole round on the device, eager and graph-captured
        c = W.edit_bs4(temperature=0.0, probabilistic=False, edit_rates=[RATES[rank]] * 4)
        ng = O.ngram_propose(c["hist"], c["hist_len"], c["n_min"], c["n_max"], c["L"], c["copy_cap"])
        lay = O.price_and_allocate(c["d"], c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len,
                                   c["coef"], c["lam"], c["budget"], c["max_verify_len"], c["policy"],
                                   c["draft_greedy"])
        logits = W.compact_logits(c, lay.row_off, lay.verify_len)
        o = O.verify_chain(logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass)
        rnd = ChainRound(c["B"], c["hist"].shape[1], c["K"], c["L"], c["V"], torch.bfloat16, logits.shape[0],
                         c["coef"], c["n_min"], c["n_max"])
        rnd.load(c["hist"], c["hist_len"], c["d"], c["c"], c["d_len"])
        rnd.logits.copy_(logits_dev(logits))
        rnd.capture(lam=c["lam"], budget=c["budget"], max_verify_len=c["max_verify_len"])
        for step in range(STEPS):
            dist.barrier()
            rnd.out_tokens.fill_(-9)
            if step % 2 == 0:
                rnd.run(c["lam"], c["budget"], c["max_verify_len"])
            else:
                rnd.graph.replay()
            torch.cuda.synchronize()
            assert np.array_equal(rnd.row_off.cpu().numpy(), lay.row_off), step
            assert np.array_equal(rnd.out_tokens.cpu().numpy(), o.out_tokens), step
            assert rnd.ws.status() == 0
            checked += 1
        # sampled with draft distributions (draws, and max(0, p - q) draws)
        c = W.edit_bs4(temperature=1.0, probabilistic=True, edit_rates=[RATES[rank]] * 4)
        ng = O.ngram_propose(c["hist"], c["hist_len"], c["n_min"], c["n_max"], c["L"], c["copy_cap"])
        lay = O.price_and_allocate(c["d"], c["c"], c["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree, ng.copy_len,
                                   c["coef"], c["lam"], c["budget"], c["max_verify_len"], c["policy"],
                                   c["draft_greedy"])
        logits = W.compact_logits(c, lay.row_off, lay.verify_len)
        ws = S.Workspace(c["B"], int(lay.row_off[-1]), c["K"], c["V"])
        lt, dt = logits_dev(logits), logits_dev(c["draft_logits"])
        for step in range(STEPS):
            dist.barrier()
            g = gpu_chain(S, ws, None, lay.row_off, lay.chain, lay.verify_len, lay.point_mass, c["draft_logits"],
                          1.0, seed=rank, step=step, logits_t=lt, draft_t=dt)
            ov = O.verify_chain(logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass, c["draft_logits"],
                                1.0, rank, step)
            compare_sampled(g, ov, logits, lay.row_off, lay.chain, lay.verify_len, lay.point_mass,
                            c["draft_logits"], 1.0)
            assert ws.status() == 0
            checked += 1
        ok = 1
    except Exception:  # reported through the file, so the other process is not left waiting
        import traceback

        ok = 0
        with open(os.path.join(outdir, f"err{rank}.txt"), "w") as f:
            f.write(traceback.format_exc())
    finally:
        with open(os.path.join(outdir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ok} {checked}")
        dist.destroy_process_group()


def test_two_processes_share_one_gpu(orc, tmp_path):
    import speculative_decoding_draft_spec_gb300 as S

    S.build()  # once, here (and the oracle, by its fixture): the children only load the libraries
    world = 2
    mp.spawn(_child, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        ok, checked = open(tmp_path / f"rank{r}.txt").read().split()
        err = (tmp_path / f"err{r}.txt")
        assert ok == "1", err.read_text() if err.exists() else "no result"
        assert int(checked) == 2 * STEPS
