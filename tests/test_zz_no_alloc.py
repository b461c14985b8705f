"""fmm_morton_keys_noalloc, the entry point for callers that cannot allocate
device memory: code that owns a fixed device budget handed out by its own
allocator, a library embedded in a host application that forbids device
allocation after start-up, or a real-time loop that must not take the
driver's allocation locks.

Its keys must equal those of the plan path (fmm_eval's sorted keys mapped back
through the sort permutation), bit for bit, on two calls in a row; the second
call checks that the shared scratch is reset between calls. This file is
collected last so that a failure here comes after every other test has run."""
import numpy as np
import pytest

from body_forces_morton_b300 import workloads as W

pytestmark = pytest.mark.gpu


def plan_keys(pos, mass, dtype):
    """Keys in the caller's order from the existing entry point."""
    import torch

    from body_forces_morton_b300 import native

    n = len(mass)
    with native.Plan(n, 4, 0.7, 64, dtype) as pl:
        tp = torch.from_numpy(pos).cuda()
        tm = torch.from_numpy(mass).cuda()
        acc = torch.empty_like(tp)
        pl.eval(tp, tm, acc, None, stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        keys_sorted = pl.export("keys")
        perm = pl.export("perm").astype(np.int64)
    out = np.empty(n, dtype=np.uint64)
    out[perm] = keys_sorted
    return out


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_noalloc_keys_equal_plan_keys_twice(dtype):
    import torch

    from body_forces_morton_b300 import native

    dt_code = native.FMM_F32 if dtype == "f32" else native.FMM_F64
    for cfg, n in ((4, 200003), (2, 77777)):  # two calls in a row, different inputs
        g = W.generate(W.WORKLOADS[cfg], n=n, dtype=dtype)
        want = plan_keys(g["pos"], g["mass"], dtype)
        tp = torch.from_numpy(g["pos"]).cuda()
        keys = torch.empty(n, dtype=torch.int64, device="cuda")
        box = torch.empty(4, dtype=torch.float64, device="cuda")
        native.fmm_morton_keys_noalloc(tp, n, dt_code, keys, box, stream=torch.cuda.current_stream())
        got = keys.cpu().numpy().view(np.uint64)
        assert np.array_equal(got, want)
        assert np.array_equal(box.cpu().numpy(), expected_box(g["pos"]))


def expected_box(pos):
    """Lower corner and side of the root cube; the side is 1 when every point coincides."""
    lo = pos.min(axis=0)
    side = (pos.max(axis=0) - lo).max()
    return np.array([*lo, side if side > 0 else 1.0], dtype=np.float64)


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("n", [1, 1 << 21])
def test_noalloc_edges(dtype, n):
    """The capacity edge (n = 2^21: every one of the 1024 partial-box slots is
    used) and a single particle (a degenerate box whose side falls back to 1)."""
    import torch

    from body_forces_morton_b300 import native

    dt_code = native.FMM_F32 if dtype == "f32" else native.FMM_F64
    g = W.generate(W.WORKLOADS[4], n=n, dtype=dtype)
    want = plan_keys(g["pos"], g["mass"], dtype)
    tp = torch.from_numpy(g["pos"]).cuda()
    keys = torch.empty(n, dtype=torch.int64, device="cuda")
    box = torch.empty(4, dtype=torch.float64, device="cuda")
    native.fmm_morton_keys_noalloc(tp, n, dt_code, keys, box, stream=torch.cuda.current_stream())
    assert np.array_equal(keys.cpu().numpy().view(np.uint64), want)
    assert np.array_equal(box.cpu().numpy(), expected_box(g["pos"]))


def test_noalloc_rejects_too_many_particles():
    import torch

    from body_forces_morton_b300 import native

    tp = torch.zeros(8, 3, dtype=torch.float32, device="cuda")
    keys = torch.empty(8, dtype=torch.int64, device="cuda")
    with pytest.raises(native.FmmError) as ei:
        native.fmm_morton_keys_noalloc(tp, (1 << 21) + 1, native.FMM_F32, keys)
    assert ei.value.status == 1
