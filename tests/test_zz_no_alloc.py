"""ssd_forward_noalloc (the allocation-free forward pass, working in the
library's fixed device scratch array) against ssd_forward on the same inputs.

Both calls run the same kernels on the same split of the work, so their
results must be identical bit for bit (a tolerance could hide a partly stale
read of the shared scratch); each case makes two calls in a row with
different inputs, so anything one call left in the scratch that the next one
read would show.  The file sorts last so that it also runs after every other
GPU test has used the library.
"""
import pytest
import torch

from state_space_sequence_ssd_gb300 import inputs as I

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def ssd():
    from state_space_sequence_ssd_gb300 import build
    build.build()
    import state_space_sequence_ssd_gb300 as m
    return m


def same(name, got, ref):
    assert bool(torch.isfinite(got.float()).all()), f"{name}: non-finite values"
    if not torch.equal(got, ref):
        err = (got.double() - ref.double()).abs()
        raise AssertionError(f"{name}: {(err > 0).sum().item()} elements differ, max |diff| {err.max().item()}")


def dev_inputs(w, seed, init):
    inp = I.make_inputs(w, seed)
    if init and inp["init"] is None:
        g = torch.Generator().manual_seed(seed + 99)
        inp["init"] = 0.1 * torch.randn((w.batch, w.nheads, w.headdim, w.dstate), generator=g)
    return {k: (None if v is None else v.cuda()) for k, v in inp.items()}


def run_pair(ssd, w, chunk_size, seed, init):
    d = dev_inputs(w, seed, init)
    y_ref, fin_ref = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], chunk_size)
    y = torch.full_like(d["x"], float("nan"))
    fin = torch.full_like(fin_ref, float("nan"))
    ssd.ssd_forward_noalloc(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], chunk_size, y, fin)
    torch.cuda.synchronize()
    assert ssd.ssd_get_device_error() == 0
    same(f"{w.name} y", y, y_ref)
    same(f"{w.name} final_state", fin, fin_ref)


CASES = [("tiny_L512_N64", 64, False), ("tiny_L512_N64", 64, True), ("mamba2_1p3b_layer_2x4096_N128", 256, False),
         ("state_sweep_L16384_N64", 128, True)]


@pytest.mark.parametrize("name,chunk_size,init", CASES)
def test_noalloc_matches_forward_twice(ssd, name, chunk_size, init):
    w = I.WORKLOADS[name]
    run_pair(ssd, w, chunk_size, seed=11, init=init)
    run_pair(ssd, w, chunk_size, seed=12, init=init)


def test_noalloc_small_after_large(ssd):
    """A small call right after a large one reuses the start of the scratch."""
    run_pair(ssd, I.WORKLOADS["mamba2_1p3b_layer_2x4096_N128"], 256, seed=21, init=True)
    run_pair(ssd, I.WORKLOADS["tiny_L512_N64"], 64, seed=22, init=False)


def test_noalloc_rejects_oversize(ssd):
    """65536 tokens x 32 heads x dstate 128 needs about 85 MiB of the 64 MiB scratch."""
    w = I.WORKLOADS["long_L65536_N128"]
    b, L, H, P, G, N = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate
    x = torch.zeros((b, L, H, P), dtype=torch.bfloat16, device="cuda")
    dt = torch.zeros((b, L, H), device="cuda")
    A = torch.zeros((H,), device="cuda")
    B = torch.zeros((b, L, G, N), dtype=torch.bfloat16, device="cuda")
    y = torch.full_like(x, 7.0)
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_forward_noalloc(x, dt, A, B, B, None, None, w.chunk_size, y)
    assert e.value.status == 6 and "SCRATCH_TOO_SMALL" in str(e.value)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all()), "a rejected call must launch nothing"
