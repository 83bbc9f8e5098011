"""The head-partitioned multi-GPU split, without a GPU: the partition planner (ssd_partition_heads)
covers every head exactly once, in whole B/C groups when there are enough groups, in blocks of two
heads otherwise; ranks of a gloo process group agree on a plan with no gaps or overlaps; and
ssd_forward_heads rejects a bad head range before touching the device."""
import itertools
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from state_space_sequence_ssd_gb300 import _ffi


@pytest.fixture(scope="module")
def ssd():
    from state_space_sequence_ssd_gb300 import build
    build.build()
    import state_space_sequence_ssd_gb300 as m
    return m


def plan(ssd, H, G, n):
    return [ssd.ssd_partition_heads(H, G, n, p) for p in range(n)]


SHAPES = [(H, G) for H in (1, 2, 3, 4, 6, 8, 12, 16, 32, 64, 80) for G in (1, 2, 3, 4, 8, 16) if H % G == 0]


@pytest.mark.parametrize("H,G", SHAPES)
def test_parts_tile_the_heads(ssd, H, G):
    hpg = H // G
    for n in (1, 2, 3, 4, 5, 8):
        parts = plan(ssd, H, G, n)
        # contiguous, in order, every head exactly once
        pos = 0
        for b, c in parts:
            assert b == pos and c >= 0
            pos += c
        assert pos == H
        if G >= n:  # whole groups, as balanced as the groups allow
            for b, c in parts:
                assert b % hpg == 0 and c % hpg == 0 and c > 0
            sizes = [c // hpg for _, c in parts]
            assert max(sizes) - min(sizes) <= 1
        elif hpg % 2 == 0:  # blocks of two heads: compute_out keeps two heads per CTA
            for b, c in parts:
                assert b % 2 == 0 and c % 2 == 0
            blocks = [c // 2 for _, c in parts]
            assert max(blocks) - min(blocks) <= 1
        else:
            sizes = [c for _, c in parts]
            assert max(sizes) - min(sizes) <= 1


def test_planner_rejects_bad_arguments(ssd):
    lib = _ffi.lib()
    import ctypes
    hb, hc = ctypes.c_int(0), ctypes.c_int(0)
    for args in ((0, 1, 1, 0), (8, 3, 2, 0), (8, 2, 0, 0), (8, 2, 2, 2), (8, 2, 2, -1), (8, 0, 2, 0)):
        assert lib.ssd_partition_heads(*args, ctypes.byref(hb), ctypes.byref(hc)) == _ffi.SSD_ERR_INVALID_ARG
    assert lib.ssd_partition_heads(8, 2, 2, 0, None, ctypes.byref(hc)) == _ffi.SSD_ERR_INVALID_ARG


FAKE = 4096


def heads_call(lib, head_begin, head_count, nheads=8):
    return lib.ssd_forward_heads(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 512, nheads, 64, 2, 64, 64,
                                 head_begin, head_count, FAKE, FAKE, None)


@pytest.mark.parametrize("hb,hc", [(-1, 2), (0, 0), (7, 2), (8, 1), (0, 9), (3, -1)])
def test_forward_heads_rejects_bad_ranges(ssd, hb, hc):
    assert heads_call(_ffi.lib(), hb, hc) == _ffi.SSD_ERR_INVALID_ARG


def test_forward_heads_shares_forward_validation(ssd):
    lib = _ffi.lib()
    # a valid range with an invalid shape (nheads % ngroups != 0) or a misaligned x is refused too
    assert lib.ssd_forward_heads(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 512, 7, 64, 2, 64, 64, 0, 2,
                                 FAKE, FAKE, None) == _ffi.SSD_ERR_INVALID_ARG
    assert lib.ssd_forward_heads(FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 512, 8, 64, 2, 64, 64, 0, 2,
                                 FAKE, FAKE, None) == _ffi.SSD_ERR_INVALID_ARG


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, shapes, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import state_space_sequence_ssd_gb300 as ssd
    res = []
    for H, G in shapes:
        b, c = ssd.ssd_partition_heads(H, G, world, rank)
        t = torch.tensor([b, c], dtype=torch.int64)
        g = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(g, t)
        res.append([tuple(int(v) for v in x) for x in g])
    if rank == 0:
        out.put(res)
    dist.destroy_process_group()


def test_ranks_agree_on_a_complete_plan():
    """Two gloo ranks each ask for their own part and gather all parts: the parts tile every shape's heads."""
    from state_space_sequence_ssd_gb300 import build
    build.build()
    shapes = [(32, 1), (32, 8), (64, 1), (12, 3), (6, 6), (1, 1)]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, shapes, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for (H, G), parts in zip(shapes, res):
        covered = list(itertools.chain.from_iterable(range(b, b + c) for b, c in parts))
        assert covered == list(range(H)), (H, G, parts)
