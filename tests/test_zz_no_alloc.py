"""verify_attn_paged_noalloc: the entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc: a plugin running inside a serving engine
whose allocator has already claimed nearly all device memory for its KV pool,
or code on a latency-critical path where cudaMalloc / cudaFree would
synchronise the device.  For them the library keeps one fixed scratch array in
device memory and this entry point uses it instead of a caller workspace.

The test calls the new entry point through the C ABI twice in a row, with
different inputs, and checks each result against the regular
verify_attn_paged on the same inputs and against the fp64 oracle, with the
tolerance of the other parity tests.  It runs alone in a fresh process or
after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_speculative_decode_gb300 as m
    m.build()
    m.init()
    return m


def _close(a_out, a_lse, b_out, b_lse):
    d = (a_out.float() - b_out.float()).abs()
    assert d.max().item() <= _gpu.OUT_MAX_ABS
    assert d.mean().item() <= _gpu.OUT_MEAN_ABS
    assert (a_lse - b_lse).abs().max().item() <= _gpu.LSE_ABS


def test_noalloc_matches_paged_on_two_calls_in_a_row(va):
    specs = [synth.Spec("na1", B=1, H=8, T=16, prefix=[4096], num_slots=1 << 16, seed=71),
             synth.Spec("na2", B=2, H=8, T=12, prefix=[1500, 333], num_slots=1 << 16, seed=72)]
    for s in specs:
        w = synth.make(s)
        d = _gpu.to_device(w)
        ref_out, ref_lse = _gpu.run(va, d, w)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        va.verify_attn_paged_noalloc(d["q"], d["kv_pool"], d["slot_idx"], d["kv_indptr"],
                                     d["prefix_len"], d["parents"], sm_scale=s.sm_scale,
                                     out=out, lse=lse)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        _close(out, lse, ref_out, ref_lse)
        ref_o, ref_l = _gpu.reference(w)
        _gpu.compare(out, lse, ref_o, ref_l)


def test_noalloc_lowers_the_automatic_split_count_to_fit(va):
    """Eight requests at H=64, T=16 (8192 query rows): the automatic split
    count's partials would not fit the scratch array, so the call lowers the
    count until they do; its result still matches the regular call (which
    keeps the automatic count) and the oracle."""
    s = synth.Spec("na4", B=8, H=64, T=16, prefix=[1100, 64, 2900, 700, 0, 1500, 333, 2048],
                   num_slots=1 << 15, seed=74)
    auto = va.auto_nsplit(s.B, s.T, s.H)
    assert va.workspace_bytes(s.B, s.T, s.H, auto) > va.NOALLOC_SCRATCH_BYTES
    w = synth.make(s)
    d = _gpu.to_device(w)
    ref_out, ref_lse = _gpu.run(va, d, w)
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        va.verify_attn_paged_noalloc(d["q"], d["kv_pool"], d["slot_idx"], d["kv_indptr"],
                                     d["prefix_len"], d["parents"], sm_scale=s.sm_scale,
                                     out=out, lse=lse)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)
    rows = _gpu.sample_rows(w, 256, seed=5)
    ref_o, ref_l = _gpu.reference(w, rows=rows)
    _gpu.compare(out, lse, ref_o, ref_l, rows=rows)


def test_noalloc_rejects_sizes_beyond_its_scratch(va):
    s = synth.Spec("na3", B=1, H=64, T=64, prefix=[100], num_slots=4096, seed=73)
    w = synth.make(s)
    d = _gpu.to_device(w)
    out = torch.empty(s.T, s.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(s.T, s.H, dtype=torch.float32, device="cuda")
    big = 1
    while va.workspace_bytes(1, s.T, s.H, big) <= va.NOALLOC_SCRATCH_BYTES:
        big += 1
    with pytest.raises(va.VaError) as e:
        va.verify_attn_paged_noalloc(d["q"], d["kv_pool"], d["slot_idx"], d["kv_indptr"],
                                     d["prefix_len"], d["parents"], sm_scale=s.sm_scale,
                                     nsplit=big, out=out, lse=lse)
    assert e.value.code == -4


def test_noalloc_rejects_sizes_whose_single_split_does_not_fit(va):
    """32768 query rows: one split's partials alone exceed the scratch array,
    so even the automatic split count cannot fit and the call is refused
    before any launch."""
    B, T, H = 4, 64, 128
    assert va.workspace_bytes(B, T, H, 1) > va.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B * T, H, 576, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4096, 576, dtype=torch.bfloat16, device="cuda")
    slots = torch.arange(B * (T + 10), dtype=torch.int32, device="cuda")
    indptr = torch.arange(0, B * (T + 10) + 1, T + 10, dtype=torch.int32, device="cuda")
    prefix = torch.full((B,), 10, dtype=torch.int32, device="cuda")
    parents = torch.full((B, T), -1, dtype=torch.int32, device="cuda")
    out = torch.empty(B * T, H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B * T, H, dtype=torch.float32, device="cuda")
    with pytest.raises(va.VaError) as e:
        va.verify_attn_paged_noalloc(q, pool, slots, indptr, prefix, parents,
                                     sm_scale=0.1, out=out, lse=lse)
    assert e.value.code == -4
