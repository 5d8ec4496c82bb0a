"""bsa_build_mask_noalloc: the mask builder for callers that cannot allocate device
memory (a framework that owns all device memory from start-up on, or a process
whose memory budget is frozen while it serves).

Its scratch is a fixed array inside the library, so the call needs no workspace.
This file is collected last on purpose: a run that stops at the first failure has
already run every other test. It must pass alone in a fresh process and after the
other tests, which both exercise the per-device set-up and the reuse of the array.
"""
import warnings

import numpy as np
import pytest
import torch

from block_sparse_attention_mean_gb300 import binding as bb
from block_sparse_attention_mean_gb300 import build as bbuild
from block_sparse_attention_mean_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bbuild.build()
    bb.load()


def _upload(inp, name):
    return torch.from_numpy(inp[name + "_bits"].view(np.int16)).cuda().view(torch.bfloat16)


def _index_buffers(w, cap):
    nB = w.N // w.block
    W = (nB + 31) // 32
    return (torch.full((w.B * w.H * nB + 1,), -1, dtype=torch.int32, device="cuda"),
            torch.full((cap,), -1, dtype=torch.int32, device="cuda"),
            torch.full((w.B * w.H * nB * W,), -1, dtype=torch.int32, device="cuda"))


def _compare_two_calls(w, q, k, spec):
    """The no-alloc builder must reproduce the workspace builder, call after call."""
    ref = bb.build_mask(q, k, w.block, density=w.density, spec=spec, shape=(w.B, w.H, w.N, w.d))
    cap = bb.bsa_mask_nnz(w.B, w.H, w.N, w.block, w.density, spec)
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for _ in range(2):
        row_ptr, col_idx, bitmap = _index_buffers(w, cap)
        bb.bsa_build_mask_noalloc(q, k, bb.BF16, w.B, w.H, w.N, w.d, w.block, w.density, spec, row_ptr,
                                  col_idx, cap, bitmap, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == bb.OK
        assert torch.equal(row_ptr, ref.row_ptr)
        assert torch.equal(col_idx[:ref.nnz], ref.col_idx[:ref.nnz])
        assert torch.equal(bitmap, ref.bitmap)


def test_noalloc_dynamic_topk_matches_workspace_builder():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=4, N=4096)
    inp = wl.make_inputs(w)
    _compare_two_calls(w, _upload(inp, "q"), _upload(inp, "k"), None)


def test_noalloc_static_band_matches_workspace_builder():
    w = wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=4)
    _compare_two_calls(w, None, None, bb.band_spec(w.n_text_blocks, w.band, list(w.anchors)))


def test_noalloc_reports_device_status():
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=1, N=1024)
    inp = wl.make_inputs(w)
    q, k = _upload(inp, "q"), _upload(inp, "k")
    q[0, 0, 7, 5] = float("nan")
    cap = bb.bsa_mask_nnz(w.B, w.H, w.N, w.block, w.density, None)
    row_ptr, col_idx, bitmap = _index_buffers(w, cap)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bb.bsa_build_mask_noalloc(q, k, bb.BF16, w.B, w.H, w.N, w.d, w.block, w.density, None, row_ptr, col_idx,
                              cap, bitmap, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == bb.ERR_NONFINITE
    # the next call starts from a cleared status word
    q[0, 0, 7, 5] = 0.0
    bb.bsa_build_mask_noalloc(q, k, bb.BF16, w.B, w.H, w.N, w.d, w.block, w.density, None, row_ptr, col_idx,
                              cap, bitmap, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == bb.OK


def test_noalloc_rejects_problems_larger_than_its_scratch():
    # 2 x B*H*nB*d*4 bytes of pooled blocks: here 2 * 64 * 1024 * 128 * 4 = 64 MiB > 16 MiB
    B, H, N, d, block = 1, 64, 65536, 128, 64
    assert bb.bsa_workspace_size(0, B, H, N, d, block) > bb.NOALLOC_SCRATCH_BYTES
    with pytest.raises(bb.BsaError) as e:
        bb.bsa_build_mask_noalloc(1 << 20, 1 << 20, bb.BF16, B, H, N, d, block, 0.1, None, 1 << 20, 1 << 20,
                                  1 << 30, 1 << 20)
    assert e.value.code == bb.ERR_WORKSPACE


def _captures_nothing(fn) -> bool:
    """Capture fn(stream) into a CUDA graph; True when the graph came out empty (torch
    warns about an empty capture)."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with warnings.catch_warnings(record=True) as rec:
        warnings.simplefilter("always")
        with torch.cuda.graph(g, stream=side):
            fn(side)
    torch.cuda.synchronize()
    return any("graph is empty" in str(r.message).lower() for r in rec)


def test_noalloc_failed_call_enqueues_nothing():
    """A call rejected by an argument check enqueues no work: captured into a CUDA graph
    on its own, it leaves the graph empty (no clearing of the array's header, no copy of a
    status word, no kernel). A valid call, captured the same way, does not."""
    w = wl.scaled(wl.WORKLOADS["dynamic_topk"], H=1, N=1024)
    inp = wl.make_inputs(w)
    q, k = _upload(inp, "q"), _upload(inp, "k")
    cap = bb.bsa_mask_nnz(w.B, w.H, w.N, w.block, w.density, None)
    row_ptr, col_idx, bitmap = _index_buffers(w, cap)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call(stream, density=w.density, rp=row_ptr, capacity=cap):
        bb.bsa_build_mask_noalloc(q, k, bb.BF16, w.B, w.H, w.N, w.d, w.block, density, None, rp, col_idx,
                                  capacity, bitmap, device_status=status, stream=stream)

    call(None)  # the per-device set-up happens outside any capture
    torch.cuda.synchronize()
    assert not _captures_nothing(call)  # control: a valid call is captured
    codes = []

    def failing(stream):
        for kw in (dict(density=float("nan")), dict(density=1.5), dict(capacity=cap - 1), dict(rp=0)):
            try:
                call(stream, **kw)
                codes.append(bb.OK)
            except bb.BsaError as e:
                codes.append(e.code)

    assert _captures_nothing(failing)
    assert codes == [bb.ERR_INVALID_ARG, bb.ERR_INVALID_ARG, bb.ERR_CAPACITY, bb.ERR_INVALID_ARG]


def test_noalloc_static_spec_sized_by_the_static_path():
    """A static build needs only per-row counts and one head's pattern, so a band
    mask whose dynamic build would not fit the array is accepted."""
    w = wl.scaled(wl.WORKLOADS["t2i_static"], B=1, H=64)
    spec = bb.band_spec(w.n_text_blocks, w.band, list(w.anchors))
    B, H, N, d, block = 1, 64, 65536 + w.n_text_blocks * 64, 128, 64
    assert bb.bsa_workspace_size(0, B, H, N, d, block) > bb.NOALLOC_SCRATCH_BYTES
    nB = N // block
    cap = bb.bsa_mask_nnz(B, H, N, block, 0.0, spec)
    row_ptr = torch.empty(B * H * nB + 1, dtype=torch.int32, device="cuda")
    col_idx = torch.empty(cap, dtype=torch.int32, device="cuda")
    bitmap = torch.empty(B * H * nB * ((nB + 31) // 32), dtype=torch.int32, device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    bb.bsa_build_mask_noalloc(None, None, bb.BF16, B, H, N, d, block, 0.0, spec, row_ptr, col_idx, cap, bitmap,
                              device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == bb.OK
    ref = bb.build_mask(None, None, block, spec=spec, shape=(B, H, N, d))
    assert torch.equal(row_ptr, ref.row_ptr)
    assert torch.equal(col_idx, ref.col_idx[:cap])
    assert torch.equal(bitmap, ref.bitmap)
