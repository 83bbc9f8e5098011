"""bench.py's multi-rank host logic on CPU: world size 2 over gloo.

Every rank times its own replica; the reported time is the slowest rank's,
so `max_over_ranks` must return the maximum on every rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(values[rank], dist, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    values = [3.5, 7.25]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == pytest.approx(7.25) and out[1] == pytest.approx(7.25)


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(2.0, None, torch.device("cpu")) == 2.0


def test_algorithmic_bytes_of_the_headline_workload():
    """bench.py's per-launch bytes at L 65536, H 32, N 128 for the library's plan of that shape (7-chunk
    spans, compute_out runs of four spans).  The roofline credits compulsory bytes only: chunk_scan's are
    x + y + B + C = 570.4 MB; the intermediates it also moves (dA_cumsum and dt rows, run-start states) are
    reported apart."""
    import bench
    from state_space_sequence_ssd_gb300 import inputs as I
    w = I.WORKLOADS["long_L65536_N128"]
    plan = {"span_chunks": 7, "scan_step": 4}
    kb = {k: bench.kernel_bytes(k, w, plan) for k in ("chunk_cumsum", "chunk_state", "state_passing", "chunk_scan")}
    mb = {k: v["compulsory"] / 1e6 for k, v in kb.items()}
    assert round(mb["chunk_scan"], 1) == 570.4
    assert round(mb["chunk_state"], 1) == 268.4
    assert round(mb["chunk_cumsum"], 1) == 41.9
    assert round(mb["state_passing"], 1) == 2.1
    tot = {k: (v["compulsory"] + v["intermediate"]) / 1e6 for k, v in kb.items()}
    assert round(tot["chunk_scan"], 1) == 597.7
    assert round(tot["chunk_cumsum"], 1) == 92.3
    assert bench.kernel_alg_bytes("chunk_scan", w, plan) == kb["chunk_scan"]["compulsory"]
    # the compulsory bytes of the kernels add up to the pass's (each input read and output written once)
    assert sum(mb.values()) * 1e6 == pytest.approx(bench.compulsory_bytes(w) + 268435456 + 2 * 16777216, rel=1e-6)


def test_source_key_ignores_comments_only():
    import bench
    assert bench._code_only("x = a; // note\n/* block\n comment */ y = b;") == bench._code_only("x = a;\ny = b;")
    assert bench._code_only("x = a;") != bench._code_only("x = b;")


def test_head_split_places_each_ranks_inputs():
    """bench.py's multi-GPU layout (on CPU tensors): world x H heads in world x G groups, rank r owning
    heads [r H, (r + 1) H) and groups [r G, (r + 1) G), with its own seeded inputs in that slice."""
    import bench
    import state_space_sequence_ssd_gb300 as ssd
    from state_space_sequence_ssd_gb300 import build, inputs as I
    build.build()
    w = I.Workload("split", 1, 96, 4, 64, 64, 2, 64, True)
    for world in (2, 3):
        for rank in range(world):
            d = I.make_inputs(w, seed=rank)
            sp = bench.head_split(w, world, rank, d, torch.device("cpu"), ssd)
            t = sp["t"]
            hb, hc = sp["head_begin"], sp["head_count"]
            assert (hb, hc) == (rank * w.nheads, w.nheads)
            assert t["x"].shape[2] == world * w.nheads and t["B"].shape[2] == world * w.ngroups
            assert torch.equal(t["x"][:, :, hb:hb + hc], d["x"])
            assert torch.equal(t["B"][:, :, rank * w.ngroups:(rank + 1) * w.ngroups], d["B"])
            assert torch.equal(t["init"][:, hb:hb + hc], d["init"])
            assert torch.equal(t["A"][hb:hb + hc], d["A"])
