"""The entry point for callers that cannot allocate device memory.

muon_ns_batched_static takes no workspace: it runs in a fixed scratch array
compiled into the library.  Its output must match muon_ns_batched with a
caller workspace, on consecutive calls (the array keeps the previous call's
contents), and problems too large for the array must be refused up front.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

TOL_BF16 = 2e-2
TOL_FP32 = 1e-4


def _rel(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return (a - b).norm().item() / max(b.norm().item(), 1e-300)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice():
    import newton_schulz_04_gb300 as m
    m.load(build_if_missing=True)
    cases = [
        (torch.bfloat16, (3, 256, 512), 71, TOL_BF16),
        (torch.bfloat16, (2, 512, 256), 72, TOL_BF16),  # second call, different shape and data
        (torch.float32, (2, 128, 256), 73, TOL_FP32),
    ]
    for dtype, (B, rows, cols), seed, tol in cases:
        X = torch.stack([synth.random_matrix(rows, cols, seed=seed + i) for i in range(B)]).to(dtype).cuda()
        ref = m.ns_batched(X, steps=5)           # caller workspace
        got = m.ns_batched_static(X, steps=5)    # fixed scratch, no allocation
        torch.cuda.synchronize()
        for i in range(B):
            assert _rel(got[i], ref[i]) < tol
        # same kernels, same order: the results agree exactly
        assert torch.equal(got, ref)


@pytest.mark.gpu
def test_static_scratch_seeded_fuzz():
    """30 seeded problems that fit the scratch (random shapes up to 700, both
    dtypes, 1-12 steps, AUTO), one after another: each equals the workspace
    entry point bit for bit, and nothing is carried over between calls."""
    import newton_schulz_04_gb300 as m
    m.load(build_if_missing=True)
    lib = m.load()
    cap = lib.muon_static_scratch_bytes()
    rng = np.random.default_rng(77)
    done = 0
    while done < 30:
        a, b = (int(v) for v in rng.integers(1, 701, size=2))
        dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
        steps = int(rng.integers(1, 13))
        B = int(rng.integers(1, 4))
        if m.workspace_bytes([(a, b)] * B, steps, dtype) + 4096 > cap:
            continue
        X = torch.stack([synth.random_matrix(a, b, seed=7000 + 10 * done + i) for i in range(B)]).to(dtype).cuda()
        ref = m.ns_batched(X, steps=steps)
        got = m.ns_batched_static(X, steps=steps)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), (done, (a, b), str(dtype), steps, B)
        assert m.static_status() == 0
        done += 1


@pytest.mark.gpu
def test_static_scratch_reports_a_timed_out_wait():
    """A kernel that gives up on a bounded wait sets the static scratch's
    status word; muon_static_status reports MUON_ERR_TIMEOUT once, clears the
    word, and the next call on the same scratch is unaffected."""
    import newton_schulz_04_gb300 as m
    m.load(build_if_missing=True)
    X = torch.stack([synth.random_matrix(256, 512, seed=74 + i) for i in range(2)]).to(torch.bfloat16).cuda()
    ref = m.ns_batched(X, steps=5)
    m.ns_batched_static(X, steps=5)
    assert m.static_status() == 0  # MUON_OK after a normal call
    m.debug_bounded_wait_static(2_000_000)  # ~1 ms of SM cycles; nothing arrives
    assert m.static_status() == 6  # MUON_ERR_TIMEOUT
    assert m.static_status() == 0  # read and cleared
    got = m.ns_batched_static(X, steps=5)
    torch.cuda.synchronize()
    assert m.static_status() == 0
    assert torch.equal(got, ref)


@pytest.mark.gpu
def test_static_scratch_refuses_oversized_problems_before_launch():
    import newton_schulz_04_gb300 as m
    lib = m.load(build_if_missing=True)
    cap = lib.muon_static_scratch_bytes()
    assert cap == 64 << 20
    big = 1 << 40  # never dereferenced: the size check comes first
    st = lib.muon_ns_batched_static(ctypes.c_void_p(big), 1, 4096, 4096, 5, None, ctypes.c_void_p(2 * big),
                                    0, 0, None)
    assert st == 4  # MUON_ERR_WORKSPACE
    assert "static scratch" in lib.muon_last_error().decode()


def test_static_entry_point_is_exported():
    from newton_schulz_04_gb300 import build as b
    b.build()
    import newton_schulz_04_gb300 as m
    lib = m.load()
    assert hasattr(lib, "muon_ns_batched_static")
    assert lib.muon_static_scratch_bytes() == 64 << 20
