"""Bounded device waits: a wait that runs out ends the call cleanly.

Every wait of the split-K kernel is bounded by a clock budget (about two
seconds).  The test build of the library (libverifyattn_testhooks.so, the same
sources with VA_TEST_HOOKS) adds one more bounded wait: the producer warps of
each CTA wait on a gate before their first copy.  Pointed at a device flag that
nothing sets, that wait runs out; the kernel must then set VA_STATUS_TIMEOUT,
leave every role through its abort path (no copy, product or bulk write still
in flight), free its tensor memory and return, so that the call completes and
the CUDA context stays usable.  Nothing here faults, traps or hangs: the flag
is plain device memory, and every wait involved has a limit.
"""
import ctypes
import time

import pytest
import torch

import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_speculative_decode_gb300 as va
    from mla_speculative_decode_gb300 import _builder
    va.build()
    va.init()
    th = ctypes.CDLL(_builder.build(testhooks=True))
    th.va_init.argtypes = [ctypes.c_int]
    th.va_test_set_gate.argtypes = [ctypes.c_void_p]
    th.verify_attn_paged.argtypes = va.load().verify_attn_paged.argtypes
    th.verify_attn_contiguous.argtypes = va.load().verify_attn_contiguous.argtypes
    assert th.va_init(torch.cuda.current_device()) == 0
    yield va, th
    th.va_test_set_gate(None)


# H=8: one 128-row block per request (one-SM products, clusters of two);
# H=32: 512 rows per request (two-SM products, clusters of four)
@pytest.mark.parametrize("H", [8, 32])
@pytest.mark.parametrize("layout", ["scattered", "contiguous"])
def test_wait_that_runs_out_sets_timeout_and_the_next_call_is_correct(libs, layout, H):
    va, th = libs
    s = synth.Spec("to", B=2, H=H, T=16, prefix=[3000, 700], num_slots=1 << 14, layout=layout,
                   seed=91)
    w = synth.make(s)
    d = _gpu.to_device(w)
    ws, ns = va.alloc_workspace(s.B, s.T, s.H)
    out = torch.empty(s.B * s.T, s.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(s.B * s.T, s.H, dtype=torch.float32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")      # nothing ever sets it
    if layout == "contiguous":
        args = (d["q"].data_ptr(), d["kv_pool"].data_ptr(), s.num_slots, 576,
                d["kv_start"].data_ptr(), d["prefix_len"].data_ptr(), d["parents"].data_ptr(),
                None, s.B, s.T, s.H, s.sm_scale, ns, 0, ws.data_ptr(), ws.numel(),
                out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
        fn = th.verify_attn_contiguous
    else:
        args = (d["q"].data_ptr(), d["kv_pool"].data_ptr(), s.num_slots, 576,
                d["slot_idx"].data_ptr(), d["kv_indptr"].data_ptr(), d["prefix_len"].data_ptr(),
                d["parents"].data_ptr(), None, s.B, s.T, s.H, s.sm_scale, ns, 0, ws.data_ptr(),
                ws.numel(), out.data_ptr(), lse.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
        fn = th.verify_attn_paged
    ref_o, ref_l = _gpu.reference(w)

    # 1. the gate closed: the call returns, its wait gives up within its budget
    assert th.va_test_set_gate(flag.data_ptr()) == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert fn(*args) == 0
    status = va.read_status(ws)          # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status & va.STATUS_TIMEOUT, hex(status)
    assert elapsed < 30.0, elapsed

    # 2. the context is usable: the product library's next call on the same
    # stream computes the step exactly
    o1, l1 = _gpu.run(va, d, w, nsplit=ns, workspace=ws, out=out, lse=lse)
    assert va.read_status(ws) == 0
    _gpu.compare(o1, l1, ref_o, ref_l)

    # 3. the test build with the gate open computes the same step bit for bit
    assert th.va_test_set_gate(None) == 0
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    args2 = args[:-3] + (out2.data_ptr(), lse2.data_ptr(), args[-1])
    assert fn(*args2) == 0
    assert va.read_status(ws) == 0
    assert torch.equal(out2, o1) and torch.equal(lse2, l1)
