"""Multi-rank path on the CPU: shards of a global problem, and two gloo ranks.

The scan shards over independent (sequence, head) units, so ranks exchange
no data of the scan; each rank draws its own contiguous group of sequences
of a global batch and the only collectives are the benchmark's barrier and
max-over-ranks timing.  These tests check that the shards partition the
global problem exactly (inputs and the oracle's results) and run the
timing reduction over two gloo ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _prefill_wl(batch):
    return synth.Workload("t", "prefill", batch, 40, 3, 8, 16, 2, "bf16", chunk=16, h0_std=0.1, carry=True)


def _varlen_wl(nseq):
    return synth.Workload("t", "varlen", 1, 0, 2, 8, 16, 1, "bf16", nseq=nseq, len_lo=3, len_hi=30)


def _global_varlen(nseq):
    wl = _varlen_wl(nseq)
    lens = synth.lengths(nseq, wl.len_lo, wl.len_hi, seed=wl.seed)
    wl.cu_seqlens = synth.varlen_cu_seqlens(lens)
    wl.seqlen = int(wl.cu_seqlens[-1])
    return wl


@pytest.mark.parametrize("variant", [{}, dict(ngroups=1, prologue=True)], ids=["per_head", "grouped_raw"])
@pytest.mark.parametrize("world", [2, 3])
def test_prefill_shards_concatenate_to_global(world, variant):
    glob = synth.prefill_inputs(synth.scaled(_prefill_wl(2 * world), **variant))
    parts = [synth.prefill_inputs(synth.shard(synth.scaled(_prefill_wl(2), **variant), r, world))
             for r in range(world)]
    for k in glob:
        if k in ("A", "D", "dt_bias"):  # per head: the same on every rank
            for p in parts:
                assert np.array_equal(p[k], glob[k]), k
        else:
            assert np.array_equal(np.concatenate([p[k] for p in parts], 0), glob[k]), k


@pytest.mark.parametrize("variant", [{}, dict(ngroups=1, prologue=True)], ids=["per_head", "grouped_raw"])
def test_decode_shards_concatenate_to_global(variant):
    base = synth.Workload("t", "decode", 2, 0, 3, 8, 16, 4, "bf16", h0_std=0.1, carry=True, **variant)
    glob = synth.decode_inputs(synth.scaled(base, batch=4), steps=5, first_step=3)
    parts = [synth.decode_inputs(synth.shard(base, r, 2), steps=5, first_step=3) for r in range(2)]
    for k in glob:
        if k in ("A", "D", "dt_bias"):
            assert all(np.array_equal(p[k], glob[k]) for p in parts), k
        elif k in ("h0", "prev_B", "prev_x"):
            assert np.array_equal(np.concatenate([p[k] for p in parts], 0), glob[k]), k
        else:  # [T][b]...
            assert np.array_equal(np.concatenate([p[k] for p in parts], 1), glob[k]), k


def test_varlen_shards_concatenate_to_global():
    world = 2
    glob_wl = _global_varlen(3 * world)
    glob = synth.prefill_inputs(glob_wl)
    shards = [synth.shard(_varlen_wl(3), r, world) for r in range(world)]
    parts = [synth.prefill_inputs(w) for w in shards]
    for k in ("x", "B", "C", "dt", "lam", "theta"):
        assert np.array_equal(np.concatenate([p[k] for p in parts], 1), glob[k]), k
    # each shard's sequences are the matching group of the global lengths
    glob_lens = np.diff(glob_wl.cu_seqlens)
    assert np.array_equal(np.concatenate([np.diff(w.cu_seqlens) for w in shards]), glob_lens)
    assert shards[1].tok_offset == shards[0].seqlen


def test_shard_rejects_bad_rank():
    with pytest.raises(ValueError):
        synth.shard(_prefill_wl(2), 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.shard(_prefill_wl(2), rank, world)
        inp = synth.prefill_inputs(wl)
        y, h, pB, px, _ = oracle.prefill(inp, batch=wl.batch, L=wl.seqlen, H=wl.nheads, P=wl.headdim,
                                         N=wl.dstate, R=wl.rank, dtype=wl.dtype, h0=inp["h0"],
                                         prev_B=inp["prev_B"], prev_x=inp["prev_x"], nthreads=1)
        ys = [torch.zeros(y.shape, dtype=torch.float64) for _ in range(world)]
        hs = [torch.zeros(h.shape, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(ys, torch.from_numpy(np.ascontiguousarray(y)))
        dist.all_gather(hs, torch.from_numpy(np.ascontiguousarray(h)))
        # timing: each rank reports its own time; the job's is the slowest
        t = bench.max_over_ranks(torch, dist, world, 10.0 + rank, "cpu")
        rate = bench.job_rate(wl.batch * wl.seqlen, 4, world, t)
        if rank == 0:
            np.savez(os.path.join(out_dir, "gathered.npz"), y=torch.cat(ys, 0).numpy(),
                     h=torch.cat(hs, 0).numpy(), t=t, rate=rate)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_partition_the_global_problem(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = np.load(tmp_path / "gathered.npz")
    glob_wl = _prefill_wl(2 * world)
    inp = synth.prefill_inputs(glob_wl)
    y, h, _, _, _ = oracle.prefill(inp, batch=glob_wl.batch, L=glob_wl.seqlen, H=glob_wl.nheads,
                                   P=glob_wl.headdim, N=glob_wl.dstate, R=glob_wl.rank, dtype=glob_wl.dtype,
                                   h0=inp["h0"], prev_B=inp["prev_B"], prev_x=inp["prev_x"], nthreads=1)
    # units are independent: the shards' results are the global results, bit for bit
    assert np.array_equal(got["y"], y)
    assert np.array_equal(got["h"], h)
    assert float(got["t"]) == 11.0  # max over ranks
    assert float(got["rate"]) == pytest.approx(2 * 40 * 4 * world / 11e-3)
