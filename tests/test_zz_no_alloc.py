"""spec_verify_dense_static (the allocation-free dense entry point, scratch in
a static device array) against spec_verify_dense with a caller workspace:
identical outputs on consecutive calls of different sizes, called through the
C ABI with raw device pointers.  Collected last on purpose, and independent of
every other test file, so it passes alone in a fresh process too."""
import ctypes

import numpy as np
import pytest

import rejection_sampling_gb300 as rs
from rejection_sampling_gb300 import workloads as wl


@pytest.fixture(scope="module")
def lib():
    rs.build()
    return rs.load()


def test_scratch_limit_rejected_on_host(lib):
    """Sizes whose workspace exceeds the static scratch on every path are
    refused before any CUDA call (here 4096 rows x 256 positions: even the
    single-pass kernel's per-position records need 32 MiB)."""
    P = None
    B, G, V = 4096, 255, 151936
    assert rs.workspace_size(B, G, V) > rs.SV_STATIC_SCRATCH_BYTES
    rc = lib.spec_verify_dense_static(P, P, rs.SV_BF16, P, P, P, B, G, V, P, P, P, P, P)
    assert rc == rs.SV_ERR_SCRATCH_LIMIT
    assert "static scratch" in rs.status_string(rc)
    # empty batch: no-op; bad sizes: invalid argument
    assert lib.spec_verify_dense_static(P, P, rs.SV_BF16, P, P, P, 0, 7, 1000, P, P, P, P, P) == rs.SV_OK
    assert lib.spec_verify_dense_static(P, P, rs.SV_BF16, P, P, P, 2, 3, 0, P, P, P, P, P) == rs.SV_ERR_INVALID_ARG


def _dev(torch, a, dev):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(dev)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point(lib):
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    # two calls in a row with different geometries (the second reuses the
    # array the first left behind), then the first again
    # the single-pass kernel (6 x 8 x 128256, 3 x 5 x 50000), the two-kernel
    # path (64 x 8 x 16384: more than one resident wave), and the warp-per-row
    # kernel (4096 x 32 x 33, which needs only the header)
    cases = [dict(B=6, gamma=7, V=128256, dtype="bf16", seed=11),
             dict(B=3, gamma=4, V=50000, dtype="f32", seed=12),
             dict(B=64, gamma=7, V=16384, dtype="bf16", seed=13),
             dict(B=4096, gamma=31, V=33, dtype="f32", seed=14),
             dict(B=6, gamma=7, V=128256, dtype="bf16", seed=11)]
    for cfg in cases:
        d = wl.dense_inputs(cfg["B"], cfg["gamma"], cfg["V"], dtype=cfg["dtype"], seed=cfg["seed"],
                            target_sigma=3.0, draft_noise=0.5)
        B, G, V = cfg["B"], cfg["gamma"], cfg["V"]
        dt = rs.SV_BF16 if cfg["dtype"] == "bf16" else rs.SV_F32
        tgt, drf = _dev(torch, d["target"], dev), _dev(torch, d["draft"], dev)
        ids, ua, us = (_dev(torch, d[k], dev) for k in ("draft_ids", "u_accept", "u_sample"))

        def outs():
            return (torch.full((B,), 7, dtype=torch.int32, device=dev),
                    torch.full((B, G + 1), 7, dtype=torch.int32, device=dev),
                    torch.full((B, V), 7.0, dtype=torch.float32, device=dev),
                    torch.full((B, G), 7.0, dtype=torch.float32, device=dev))

        ref, got = outs(), outs()
        ws = torch.zeros(rs.workspace_size(B, G, V), dtype=torch.uint8, device=dev)
        rc = lib.spec_verify_dense(tgt.data_ptr(), drf.data_ptr(), dt, ids.data_ptr(), ua.data_ptr(),
                                   us.data_ptr(), B, G, V, *(t.data_ptr() for t in ref),
                                   ws.data_ptr(), ws.numel(), sp)
        assert rc == rs.SV_OK
        rc = lib.spec_verify_dense_static(tgt.data_ptr(), drf.data_ptr(), dt, ids.data_ptr(),
                                          ua.data_ptr(), us.data_ptr(), B, G, V,
                                          *(t.data_ptr() for t in got), sp)
        assert rc == rs.SV_OK, rs.status_string(rc)
        torch.cuda.synchronize(dev)
        assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1]), cfg
        assert (got[0] >= 0).all()
        assert torch.equal(ref[2], got[2]) and torch.equal(ref[3], got[3]), cfg


@pytest.mark.gpu
def test_static_scratch_limit_of_the_path_taken(lib):
    """4096 rows x 16 positions x 151936: the single-pass records would fit
    the array, but the grid is many waves, so the call takes the two-kernel
    path, whose piece records do not fit: refused on the host before anything
    is launched or any pointer is touched (the pointers are never read)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    sp = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    fake = 1 << 20  # aligned, never dereferenced: the call is refused first
    B, G, V = 4096, 15, 151936
    rc = lib.spec_verify_dense_static(fake, fake, rs.SV_BF16, fake, fake, fake, B, G, V, fake, fake,
                                      None, None, sp)
    assert rc == rs.SV_ERR_SCRATCH_LIMIT, rs.status_string(rc)
