"""The layout entry point that allocates nothing (moe_expand_layout_noalloc).

Some callers cannot allocate device memory when the layer runs: a serving
engine that has reserved nearly all of HBM for its own pool, or a host loop
that must not call cudaMalloc there because it can synchronise the device.
For them the layout call takes its scratch from a fixed array inside the
library. These tests call it through the C ABI and check that it gives
exactly what the allocating entry point gives, on two calls in a row with
different inputs (the array keeps the previous call's contents), and that it
refuses sizes its array cannot hold. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from expanded_layout_expert_gb300 import build, _capi
    build.build()
    return _capi.load()


def _outputs(T, K, E, M_cap, dev):
    return dict(psum=torch.full((E,), -9, dtype=torch.int32, device=dev),
                start=torch.full((E,), -9, dtype=torch.int32, device=dev),
                total=torch.full((1,), -9, dtype=torch.int32, device=dev),
                m_indices=torch.full((M_cap,), -9, dtype=torch.int32, device=dev),
                src2dst=torch.full((T, K), -9, dtype=torch.int32, device=dev),
                tile_prefix=torch.full((E + 1,), -9, dtype=torch.int32, device=dev),
                status=torch.zeros(1, dtype=torch.int32, device=dev))


def _run(lib, which, ids, E, align, n_valid, M_cap):
    T, K = ids.shape
    o = _outputs(T, K, E, M_cap, ids.device)
    s = torch.cuda.current_stream().cuda_stream
    args = [ids.data_ptr(), T, K, E, align, n_valid.data_ptr(), M_cap, o["psum"].data_ptr(),
            o["start"].data_ptr(), o["total"].data_ptr(), o["m_indices"].data_ptr(),
            o["src2dst"].data_ptr(), o["tile_prefix"].data_ptr()]
    if which == "noalloc":
        rc = lib.moe_expand_layout_noalloc(*args, o["status"].data_ptr(), s)
    else:
        ws = torch.zeros(lib.moe_workspace_size(T, K, E), dtype=torch.uint8, device=ids.device)
        rc = lib.moe_expand_layout(*args, ws.data_ptr(), ws.numel(), o["status"].data_ptr(), s)
    assert rc == 0, lib.moe_last_error_string()
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


@pytest.mark.parametrize("names", [("zipf_t16384_h7168", "mid_padded"),
                                   ("padded_t32768_valid6000_h4096", "tiny_h512")])
def test_noalloc_layout_equals_the_allocating_call_twice_in_a_row(lib, names):
    for name in names:                      # two calls in a row, different inputs
        cfg = synth.config_by_name(name)
        d = synth.generate(cfg, device="cuda", with_weights=False)
        ids = d["topk_ids"]
        nv = torch.tensor([d["n_valid"]], dtype=torch.int32, device="cuda")
        M_cap = lib.moe_expanded_capacity(cfg.T, cfg.K, cfg.E, cfg.align)
        want = _run(lib, "ws", ids, cfg.E, cfg.align, nv, M_cap)
        got = _run(lib, "noalloc", ids, cfg.E, cfg.align, nv, M_cap)
        assert got["status"][0] == 0
        for k in ("psum", "start", "total", "m_indices", "src2dst", "tile_prefix"):
            assert np.array_equal(got[k], want[k]), (name, k)


def _launch(lib, which, ids, E, align, n_valid, M_cap, o, ws=None):
    T, K = ids.shape
    s = torch.cuda.current_stream().cuda_stream
    args = [ids.data_ptr(), T, K, E, align, n_valid.data_ptr(), M_cap, o["psum"].data_ptr(),
            o["start"].data_ptr(), o["total"].data_ptr(), o["m_indices"].data_ptr(),
            o["src2dst"].data_ptr(), o["tile_prefix"].data_ptr()]
    if which == "noalloc":
        rc = lib.moe_expand_layout_noalloc(*args, o["status"].data_ptr(), s)
    else:
        rc = lib.moe_expand_layout(*args, ws.data_ptr(), ws.numel(), o["status"].data_ptr(), s)
    assert rc == 0, lib.moe_last_error_string()


def test_noalloc_calls_queued_on_one_stream_without_a_host_wait(lib):
    """The array is shared by every call, and the contract is stream order:
    three calls with different inputs and separate outputs queued back to back
    on one stream, with no synchronisation between them, each give what the
    allocating call gives."""
    dev = "cuda"
    runs = []
    for name in ("uniform_t4096_h4096", "zipf_t16384_h7168", "mid_zipf_ragged"):
        cfg = synth.config_by_name(name)
        d = synth.generate(cfg, device=dev, with_weights=False)
        nv = torch.tensor([d["n_valid"]], dtype=torch.int32, device=dev)
        M_cap = lib.moe_expanded_capacity(cfg.T, cfg.K, cfg.E, cfg.align)
        runs.append((cfg, d["topk_ids"], nv, M_cap))
    outs = []
    for cfg, ids, nv, M_cap in runs:               # queued, no host wait in between
        o = _outputs(cfg.T, cfg.K, cfg.E, M_cap, dev)
        _launch(lib, "noalloc", ids, cfg.E, cfg.align, nv, M_cap, o)
        outs.append(o)
    torch.cuda.synchronize()
    for (cfg, ids, nv, M_cap), o in zip(runs, outs):
        want = _run(lib, "ws", ids, cfg.E, cfg.align, nv, M_cap)
        assert o["status"].item() == 0
        for k in ("psum", "start", "total", "m_indices", "src2dst", "tile_prefix"):
            assert np.array_equal(o[k].cpu().numpy(), want[k]), (cfg.name, k)


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    cap = lib.moe_expand_layout_noalloc_max_scratch()
    assert cap == 1 << 20
    E, K = 1024, 8
    T = 1 << 17                     # needs 2*1024*512*4 bytes > 1 MiB
    assert lib.moe_workspace_size(T, K, E) > cap
    small = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = small.data_ptr()
    rc = lib.moe_expand_layout_noalloc(p, T, K, E, 128, None, 64, p, p, p, p, p, p, None,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == -1
    assert b"scratch" in lib.moe_last_error_string()
