"""GPU vs fp64 oracle, element by element, through the C ABI (needs an sm_103 GPU).

Bar: out max-abs <= 2e-2 and mean-abs <= 2e-3, lse abs <= 1e-3, on the same
seeded inputs.  Integer results (defrag bytes, slot tables, status bits) are
compared exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _gpu

pytestmark = pytest.mark.gpu

PATHS = {"fma": 1, "tc": 2, "tc1sm": 3}


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_speculative_decode_gb300 as m
    m.build()
    m.init()
    return m


def _need(va, path, B, T, H):
    if path in (PATHS["tc"], PATHS["tc1sm"]):
        try:
            va.auto_nsplit(B, T, H, path)
        except va.VaError as e:
            if e.code == -5:
                pytest.skip("tensor-core path does not take this shape")
            raise


# ------------------------------------------------------------ small configs

@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
@pytest.mark.parametrize("name", ["tiny", "tp8"])
def test_config_full_parity(va, name, path):
    w = synth.make(synth.spec(name))
    s = w.spec
    _need(va, path, s.B, s.T, s.H)
    d = _gpu.to_device(w)
    out, lse = _gpu.run(va, d, w, path=path)
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out, lse, ref_o, ref_l)


SWEEP = [
    # B, H, T, prefixes, tree, nsplit
    (1, 1, 1, [0], "chain", 1),
    (1, 1, 1, [1], "chain", 4),
    (1, 8, 3, [63], "random", 2),
    (1, 8, 5, [64], "random", 3),
    (1, 8, 7, [65], "flat", 16),
    (1, 16, 16, [127], "random", 64),
    (1, 8, 16, [128], "random", 1),
    (1, 8, 16, [129], "random", 128),
    (1, 2, 64, [200], "random", 5),
    (1, 4, 64, [1000], "chain", 7),
    (3, 8, 9, [0, 300, 77], "random", 4),
    (2, 16, 4, [513, 1], "random", 0),
    (1, 64, 2, [2049], "random", 0),
    (1, 5, 13, [777], "random", 0),
    # several 128-row blocks with a ragged last one
    (1, 24, 10, [3000], "random", 0),
    (2, 40, 7, [100, 2500], "random", 3),
    (1, 128, 2, [700], "flat", 0),
    # just over one 128-row block: two-SM products whose second half is
    # mostly (129 rows) or partly (136) padding, and 1.5 units of 256 rows
    # with 40 splits of two tiles each
    (1, 43, 3, [300], "random", 0),
    (2, 8, 17, [150, 1400], "chain", 0),
    (1, 24, 16, [5000], "random", 40),
    # many short requests: the split rule's several-waves regime
    (16, 8, 4, [0, 5, 64, 65, 127, 128, 129, 300, 1, 2, 3, 511, 512, 513, 40, 90], "random", 0),
]


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
@pytest.mark.parametrize("B,H,T,prefix,tree,nsplit", SWEEP)
def test_shape_sweep(va, B, H, T, prefix, tree, nsplit, path):
    _need(va, path, B, T, H)
    seed = hash((B, H, T, tuple(prefix))) % 1000
    s = synth.Spec("sweep", B=B, H=H, T=T, prefix=prefix, num_slots=8192, tree=tree, seed=seed)
    w = synth.make(s)
    d = _gpu.to_device(w)
    out, lse = _gpu.run(va, d, w, path=path, nsplit=nsplit)
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
def test_canary_unreferenced_rows_are_nan(va, path):
    """Every pool row and padding column the step must not read holds bf16 NaN:
    a stray read poisons the output."""
    for name in ("tiny", "tp8"):
        s = synth.spec(name, canary=True, seed=synth.spec(name).seed + 100, row_stride=640,
                       num_slots=1 << 16)
        _need(va, path, s.B, s.T, s.H)
        w = synth.make(s)
        d = _gpu.to_device(w)
        out, lse = _gpu.run(va, d, w, path=path)
        ref_o, ref_l = _gpu.reference(w)
        _gpu.compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
@pytest.mark.parametrize("nsplit", [1, 3])
def test_forced_rescales(va, path, nsplit):
    """Later tiles whose scores jump far above the running maximum (the rotary
    columns of their keys are scaled by 16 and 64; values are unchanged), so
    the online softmax must move its reference and rescale the accumulator."""
    s = synth.Spec("resc", B=1, H=8, T=16, prefix=[700], num_slots=4096, seed=81)
    _need(va, path, s.B, s.T, s.H)
    w = synth.make(s)
    for (j0, j1), f in (((192, 256), 16.0), ((448, 512), 64.0)):
        rows = w.slot_idx[j0:j1].long()
        w.kv_pool[rows, 512:576] *= f
    d = _gpu.to_device(w)
    ws, _ = va.alloc_workspace(s.B, s.T, s.H, nsplit, path)
    out, lse = _gpu.run(va, d, w, path=path, nsplit=nsplit, workspace=ws)
    assert va.read_status(ws) == 0
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out, lse, ref_o, ref_l)


# -------------------------------------------- full sizes

@pytest.mark.parametrize("layout", ["scattered", "contiguous"])
def test_fullh_every_row(va, layout):
    """The full-H configuration (H=64, T=16, prefix 65536: eight 128-row
    blocks), in both layouts the benchmark times -- scattered slots and the
    contiguous (defragmented) pool read by 3-D TMA boxes -- at the automatic
    split count, compared with the oracle on every one of its 1024 rows."""
    w = synth.make(synth.spec("fullh", layout=layout))
    d = _gpu.to_device(w)
    out, lse = _gpu.run(va, d, w, path=0)
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("name", ["long", "batched"])
def test_full_size_sampled_rows(va, name):
    """The long-context and batched configurations at the benchmark's launch
    setting (automatic split count), checked on sampled rows the oracle
    evaluates one by one."""
    w = synth.make(synth.spec(name))
    d = _gpu.to_device(w)
    out, lse = _gpu.run(va, d, w, path=0)
    rows = _gpu.sample_rows(w, 256 if name == "long" else 512, seed=1)
    ref_o, ref_l = _gpu.reference(w, rows=rows)
    _gpu.compare(out, lse, ref_o, ref_l, rows=rows)


def test_batched_replayed_graph_with_new_prefixes_and_slots(va):
    """The batched configuration (8 requests, H=64, T=16, ragged prefixes in
    [1024, 65536], one shared 2^20-slot pool) captured into a CUDA graph once
    and replayed: first on its own inputs, then after new prefix lengths, slot
    tables, trees and queries of another draw were copied into the same
    buffers.  Each replay is compared with the oracle on sampled rows and with
    an eager call on the same inputs bit for bit."""
    s1 = synth.spec("batched")
    g = torch.Generator().manual_seed(4242)
    pre2 = [int(x) for x in torch.randint(1024, 65537, (s1.B,), generator=g)]
    s2 = synth.spec("batched", prefix=pre2, seed=14)
    w1 = synth.make(s1)
    w2 = synth.make(s2)
    w2.kv_pool = w1.kv_pool
    d = _gpu.to_device(w1)
    cap = max(w1.slot_idx.numel(), w2.slot_idx.numel())
    slots = torch.zeros(cap, dtype=torch.int32, device="cuda")
    slots[:w1.slot_idx.numel()] = d["slot_idx"]
    d["slot_idx"] = slots
    ws, ns = va.alloc_workspace(s1.B, s1.T, s1.H)
    rows_total = s1.B * s1.T
    out = torch.empty(rows_total, s1.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(rows_total, s1.H, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        _gpu.run(va, d, w1, nsplit=ns, workspace=ws, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _gpu.run(va, d, w1, nsplit=ns, workspace=ws, out=out, lse=lse)
    for w, seed in ((w1, 11), (w2, 12)):
        if w is w2:
            d["q"].copy_(w2.q.cuda())
            d["slot_idx"][:w2.slot_idx.numel()].copy_(w2.slot_idx.cuda())
            d["kv_indptr"].copy_(w2.kv_indptr.cuda())
            d["prefix_len"].copy_(w2.prefix_len.cuda())
            d["parents"].copy_(w2.parents.cuda())
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert va.read_status(ws) == 0
        o_rep, l_rep = out.clone(), lse.clone()
        o_eager, l_eager = _gpu.run(va, d, w, nsplit=ns)
        torch.cuda.synchronize()
        assert torch.equal(o_rep, o_eager) and torch.equal(l_rep, l_eager)
        rows = _gpu.sample_rows(w, 256, seed=seed)
        ref_o, ref_l = _gpu.reference(w, rows=rows)
        _gpu.compare(o_rep, l_rep, ref_o, ref_l, rows=rows)


def test_long_nsplit_sweep(va):
    """The long-context config at every split count of the sweep agrees with
    the oracle and with itself (splits change rounding only)."""
    w = synth.make(synth.spec("long"))
    d = _gpu.to_device(w)
    rows = _gpu.sample_rows(w, 24, seed=2)
    ref_o, ref_l = _gpu.reference(w, rows=rows)
    for ns in (16, 32, 64, 96, 128):
        out, lse = _gpu.run(va, d, w, path=0, nsplit=ns)
        _gpu.compare(out, lse, ref_o, ref_l, rows=rows)


# -------------------------------------------------------- layout variants

@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
def test_contiguous_matches_oracle_and_paged(va, path):
    s = synth.Spec("contig", B=3, H=8, T=16, prefix=[700, 64, 2000], num_slots=1 << 14,
                   layout="contiguous", seed=31)
    _need(va, path, s.B, s.T, s.H)
    w = synth.make(s)
    d = _gpu.to_device(w)
    out_c, lse_c = _gpu.run(va, d, w, path=path, layout="contiguous", nsplit=8)
    out_p, lse_p = _gpu.run(va, d, w, path=path, layout="scattered", nsplit=8)
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out_c, lse_c, ref_o, ref_l)
    assert torch.equal(out_c, out_p) and torch.equal(lse_c, lse_p)


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
@pytest.mark.parametrize("H", [8, 64])
def test_contiguous_canary_padded_rows(va, path, H):
    """Contiguous pools of 640-element rows whose padding columns, and every
    row outside the requests' ranges, hold bf16 NaN: the TMA boxes (whole
    tiles) and the copies (ragged tiles) read only the requests' rows and their
    576 columns.  H=8 runs one-SM products, H=64 two-SM products."""
    s = synth.Spec("contig_canary", B=2, H=H, T=16, prefix=[2000, 777], num_slots=1 << 13,
                   layout="contiguous", seed=91 + H, canary=True, row_stride=640)
    _need(va, path, s.B, s.T, s.H)
    w = synth.make(s)
    d = _gpu.to_device(w)
    out, lse = _gpu.run(va, d, w, path=path, layout="contiguous")
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("nsplit", [0, 3, 11])
def test_contiguous_full_h_row_blocks(va, nsplit):
    """Contiguous pools at H=64, T=16 (eight 128-row blocks per request): the
    whole 64-key tiles arrive as one 3-D TMA box, each split's ragged last tile
    by 16-byte copies; two requests with different prefix lengths (neither a
    multiple of 64).  Every row against the oracle, and bit for bit against the
    paged call on the same rows."""
    s = synth.Spec("contig_h64", B=2, H=64, T=16, prefix=[3000, 1237], num_slots=1 << 14,
                   layout="contiguous", seed=37)
    w = synth.make(s)
    d = _gpu.to_device(w)
    ws, ns = va.alloc_workspace(s.B, s.T, s.H, nsplit)
    out_c, lse_c = _gpu.run(va, d, w, layout="contiguous", nsplit=ns, workspace=ws)
    assert va.read_status(ws) == 0
    out_c, lse_c = out_c.clone(), lse_c.clone()
    out_p, lse_p = _gpu.run(va, d, w, layout="scattered", nsplit=ns)
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out_c, lse_c, ref_o, ref_l)
    assert torch.equal(out_c, out_p) and torch.equal(lse_c, lse_p)


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
def test_contiguous_many_tiles_per_split(va, path):
    """Long splits (dozens of 64-key tiles each) in the contiguous layout,
    whose whole tiles are read as boxes: the copy ring wraps many times."""
    s = synth.Spec("contig_long", B=2, H=8, T=16, prefix=[9000, 5000], num_slots=1 << 15,
                   layout="contiguous", seed=33)
    _need(va, path, s.B, s.T, s.H)
    w = synth.make(s)
    d = _gpu.to_device(w)
    for ns in (1, 2):
        ws, _ = va.alloc_workspace(s.B, s.T, s.H, ns, path)
        out, lse = _gpu.run(va, d, w, path=path, layout="contiguous", nsplit=ns, workspace=ws)
        assert va.read_status(ws) == 0
        ref_o, ref_l = _gpu.reference(w)
        _gpu.compare(out, lse, ref_o, ref_l)


def test_tree_bits_input_equals_parents(va):
    w = synth.make(synth.spec("tp8"))
    d = _gpu.to_device(w)
    bits, _ = oracle.tree_bits(w.parents.numpy())
    bits_t = torch.from_numpy(bits.view(np.int64)).cuda()
    o1, l1 = _gpu.run(va, d, w, bits=bits_t)
    o2, l2 = _gpu.run(va, d, w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_paths_agree_with_each_other(va):
    w = synth.make(synth.spec("tp8"))
    s = w.spec
    d = _gpu.to_device(w)
    o1, l1 = _gpu.run(va, d, w, path=1)
    try:
        va.auto_nsplit(s.B, s.T, s.H, 2)
    except va.VaError:
        pytest.skip("tensor-core path does not take this shape")
    o2, l2 = _gpu.run(va, d, w, path=2)
    assert (o1.float() - o2.float()).abs().max().item() <= 2 * _gpu.OUT_MAX_ABS
    assert (l1 - l2).abs().max().item() <= 2 * _gpu.LSE_ABS


# ------------------------------------------------ capture, determinism

@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
def test_graph_capture_replay_with_new_inputs(va, path):
    """Capture one call, then change prefix lengths, slots, parents and q in
    place: the replay equals a fresh eager call bit for bit."""
    s = synth.Spec("cap", B=2, H=8, T=16, prefix=[3000, 1500], num_slots=1 << 15, seed=41)
    _need(va, path, s.B, s.T, s.H)
    w1 = synth.make(s)
    w2 = synth.make(synth.Spec("cap", B=2, H=8, T=16, prefix=[2500, 2900], num_slots=1 << 15,
                               seed=42))
    w2.kv_pool = w1.kv_pool
    d = _gpu.to_device(w1)
    cap = max(w1.slot_idx.numel(), w2.slot_idx.numel())
    slots = torch.zeros(cap, dtype=torch.int32, device="cuda")
    slots[:w1.slot_idx.numel()] = d["slot_idx"]
    d["slot_idx"] = slots
    ws, ns = va.alloc_workspace(s.B, s.T, s.H, 0, path)
    out = torch.empty(s.B * s.T, s.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(s.B * s.T, s.H, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        _gpu.run(va, d, w1, path=path, nsplit=ns, workspace=ws, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _gpu.run(va, d, w1, path=path, nsplit=ns, workspace=ws, out=out, lse=lse)
    g.replay()
    torch.cuda.synchronize()
    ref1_o, ref1_l = _gpu.reference(w1)
    _gpu.compare(out, lse, ref1_o, ref1_l)
    # new step: same buffers, new contents
    d["q"].copy_(w2.q.cuda())
    d["slot_idx"][:w2.slot_idx.numel()].copy_(w2.slot_idx.cuda())
    d["kv_indptr"].copy_(w2.kv_indptr.cuda())
    d["prefix_len"].copy_(w2.prefix_len.cuda())
    d["parents"].copy_(w2.parents.cuda())
    g.replay()
    torch.cuda.synchronize()
    o_rep, l_rep = out.clone(), lse.clone()
    o_eager, l_eager = _gpu.run(va, d, w2, path=path, nsplit=ns)
    torch.cuda.synchronize()
    assert torch.equal(o_rep, o_eager) and torch.equal(l_rep, l_eager)
    ref2_o, ref2_l = _gpu.reference(w2)
    _gpu.compare(o_rep, l_rep, ref2_o, ref2_l)
    assert va.read_status(ws) == 0


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("writer", ["kernel", "copy"])
def test_inputs_written_by_the_previous_kernel(va, path, graph, writer):
    """The call's first kernel may start while the stream's previous kernel
    finishes (programmatic dependent launch) but must read no input before it
    has completed: the step's q, slots, parents and prefix lengths are written
    immediately before the call (prefix lengths last), after a call on the old
    contents -- by device kernels (elementwise multiplies by 1) or by copies
    from pinned host memory."""
    s1 = synth.Spec("pdl", B=2, H=8, T=16, prefix=[3000, 1500], num_slots=1 << 15, seed=43)
    _need(va, path, s1.B, s1.T, s1.H)
    w1 = synth.make(s1)
    w2 = synth.make(synth.Spec("pdl", B=2, H=8, T=16, prefix=[2500, 2900], num_slots=1 << 15,
                               seed=44))
    w2.kv_pool = w1.kv_pool
    d = _gpu.to_device(w1)
    cap = max(w1.slot_idx.numel(), w2.slot_idx.numel())
    slots = torch.zeros(cap, dtype=torch.int32, device="cuda")
    slots[:w1.slot_idx.numel()] = d["slot_idx"]
    d["slot_idx"] = slots
    on = "cuda" if writer == "kernel" else "cpu"
    src = {"q": w2.q.to(on), "kv_indptr": w2.kv_indptr.to(on), "parents": w2.parents.to(on),
           "prefix_len": w2.prefix_len.to(on)}
    src_slots = torch.zeros(cap, dtype=torch.int32, device=on)
    src_slots[:w2.slot_idx.numel()] = w2.slot_idx
    if writer == "copy":
        src = {k: v.pin_memory() for k, v in src.items()}
        src_slots = src_slots.pin_memory()

    def write(dst, val):
        if writer == "kernel":
            torch.mul(val, 1, out=dst)
        else:
            dst.copy_(val, non_blocking=True)
    ws, ns = va.alloc_workspace(s1.B, s1.T, s1.H, 0, path)
    out = torch.empty(s1.B * s1.T, s1.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(s1.B * s1.T, s1.H, dtype=torch.float32, device="cuda")

    def step():
        _gpu.run(va, d, w1, path=path, nsplit=ns, workspace=ws, out=out, lse=lse)
        write(d["q"], src["q"])
        write(d["slot_idx"], src_slots)
        write(d["kv_indptr"], src["kv_indptr"])
        write(d["parents"], src["parents"])
        write(d["prefix_len"], src["prefix_len"])
        _gpu.run(va, d, w2, path=path, nsplit=ns, workspace=ws, out=out, lse=lse)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        if graph:
            step()   # warm-up on the side stream before capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            # the old contents again, then one replay
            for k in ("q", "kv_indptr", "parents", "prefix_len"):
                d[k].copy_(getattr(w1, k).cuda())
            d["slot_idx"][:w1.slot_idx.numel()].copy_(w1.slot_idx.cuda())
            out.fill_(float("nan"))
            g.replay()
        else:
            step()
    torch.cuda.synchronize()
    ref_o, ref_l = _gpu.reference(w2)
    _gpu.compare(out, lse, ref_o, ref_l)
    assert va.read_status(ws) == 0


def test_deterministic(va):
    w = synth.make(synth.spec("tp8"))
    d = _gpu.to_device(w)
    o1, l1 = _gpu.run(va, d, w, nsplit=37)
    o2, l2 = _gpu.run(va, d, w, nsplit=37)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# -------------------------------------------------- guards and status

def test_guard_regions_untouched(va):
    w = synth.make(synth.spec("tiny"))
    s = w.spec
    d = _gpu.to_device(w)
    ns = 6
    n_ws = va.workspace_bytes(s.B, s.T, s.H, ns)
    G = 4096
    ws_big = torch.full((n_ws + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    rows = s.B * s.T
    out_big = torch.full((rows * s.H * 512 + 2 * G,), 7.0, dtype=torch.bfloat16, device="cuda")
    lse_big = torch.full((rows * s.H + 2 * G,), 3.0, dtype=torch.float32, device="cuda")
    ws = ws_big[G:G + n_ws]
    out = out_big[G:G + rows * s.H * 512].view(rows, s.H, 512)
    lse = lse_big[G:G + rows * s.H].view(rows, s.H)
    _gpu.run(va, d, w, nsplit=ns, workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(ws_big[:G] == 0xA5) and torch.all(ws_big[G + n_ws:] == 0xA5)
    assert torch.all(out_big[:G] == 7.0) and torch.all(out_big[G + rows * s.H * 512:] == 7.0)
    assert torch.all(lse_big[:G] == 3.0) and torch.all(lse_big[G + rows * s.H:] == 3.0)
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
def test_bad_slot_is_skipped_and_flagged(va, path):
    s = synth.Spec("bad", B=1, H=8, T=16, prefix=[300], num_slots=4096, seed=51)
    _need(va, path, s.B, s.T, s.H)
    w = synth.make(s)
    w.slot_idx[7] = 4096 + 3
    w.slot_idx[150] = -5
    d = _gpu.to_device(w)
    ws, ns = va.alloc_workspace(s.B, s.T, s.H, 0, path)
    out, lse = _gpu.run(va, d, w, path=path, nsplit=ns, workspace=ws)
    assert va.read_status(ws) & va.STATUS_BAD_SLOT
    ref_o, ref_l = _gpu.reference(w)      # the oracle skips the same keys
    _gpu.compare(out, lse, ref_o, ref_l)


def test_bad_parent_flagged(va):
    s = synth.Spec("badp", B=2, H=4, T=8, prefix=[100, 50], num_slots=4096, seed=52)
    w = synth.make(s)
    w.parents[1, 5] = 6       # not an earlier node
    d = _gpu.to_device(w)
    ws, ns = va.alloc_workspace(s.B, s.T, s.H, 0)
    out, lse = _gpu.run(va, d, w, nsplit=ns, workspace=ws)
    assert va.read_status(ws) == va.STATUS_BAD_PARENT
    ref_o, ref_l = _gpu.reference(w)      # oracle: that node hangs off the prefix
    _gpu.compare(out, lse, ref_o, ref_l)


def test_short_slot_list_flagged(va):
    s = synth.Spec("short", B=2, H=4, T=8, prefix=[100, 50], num_slots=4096, seed=53)
    w = synth.make(s)
    d = _gpu.to_device(w)
    d["prefix_len"][1] = 80   # slot list of request 1 holds only 50 + 8 keys
    ws, ns = va.alloc_workspace(s.B, s.T, s.H, 0)
    out, lse = _gpu.run(va, d, w, nsplit=ns, workspace=ws)
    assert va.read_status(ws) == va.STATUS_BAD_INDPTR
    assert torch.isfinite(out.float()).all()
    # request 0 is unaffected
    ref_o, ref_l = _gpu.reference(w)
    rows0 = s.T * s.H
    _gpu.compare(out[:s.T], lse[:s.T], ref_o[:rows0], ref_l[:rows0])


# ------------------------------------------------------------------ defrag

def test_defrag_byte_exact_and_attention_preserved(va):
    s = synth.Spec("defrag", B=3, H=8, T=16, prefix=[500, 1200, 64], num_slots=1 << 13, seed=61)
    w = synth.make(s)
    d = _gpu.to_device(w)
    # destinations: a fresh upper half of the pool that no live row uses
    extra = synth._bf16_normal((s.num_slots, 576), torch.Generator().manual_seed(62))
    w.kv_pool = torch.cat([w.kv_pool, extra])
    d["kv_pool"] = w.kv_pool.cuda()
    N = [p + s.T for p in s.prefix]
    dst, pos = [], s.num_slots + 17
    for n in N:
        dst.append(pos)
        pos += n + 5
    dst_t = torch.tensor(dst, dtype=torch.int64)
    out0, lse0 = _gpu.run(va, d, w, nsplit=4)
    pool_ref, slots_ref = oracle.defrag(synth.as_u16(w.kv_pool), w.slot_idx.numpy(),
                                        w.kv_indptr.numpy().astype(np.int64), dst_t.numpy())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    new_slots = d["slot_idx"].clone()
    va.verify_attn_defrag(d["kv_pool"], d["slot_idx"], d["kv_indptr"], dst_t.cuda(),
                          slot_idx_out=new_slots, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_pool = d["kv_pool"].cpu().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got_pool, pool_ref)
    np.testing.assert_array_equal(new_slots.cpu().numpy(), slots_ref)
    # paged over the new table and contiguous over dst_base both reproduce the step
    d["slot_idx"] = new_slots
    out1, lse1 = _gpu.run(va, d, w, nsplit=4, layout="scattered")
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    d["kv_start"] = dst_t.cuda()
    out2, lse2 = _gpu.run(va, d, w, nsplit=4, layout="contiguous")
    assert torch.equal(out0, out2) and torch.equal(lse0, lse2)


@pytest.mark.parametrize("stride", [576, 640, 1152])
def test_defrag_row_strides_byte_exact(va, stride):
    """Whole rows of any stride move byte for byte: rows of at most 96 16-byte
    chunks go through the four-rows-per-round path, wider rows through the
    chunk loop; a ragged last round of each request included."""
    n_slots = 4096
    g = torch.Generator().manual_seed(63 + stride)
    pool = synth._bf16_normal((2 * n_slots, stride), g)
    src = torch.randperm(n_slots, generator=g)[:701].to(torch.int32)
    indptr = torch.tensor([0, 303, 701], dtype=torch.int32)
    dst = torch.tensor([n_slots + 5, n_slots + 400], dtype=torch.int64)
    ref_pool, ref_slots = oracle.defrag(synth.as_u16(pool), src.numpy(),
                                        indptr.numpy().astype(np.int64), dst.numpy())
    dpool = pool.cuda()
    new_slots = src.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    va.verify_attn_defrag(dpool, src.cuda(), indptr.cuda(), dst.cuda(), slot_idx_out=new_slots,
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(dpool.cpu().view(torch.int16).numpy().view(np.uint16), ref_pool)
    np.testing.assert_array_equal(new_slots.cpu().numpy(), ref_slots)


def test_defrag_bad_rows_flagged_not_written(va):
    pool = torch.randn(256, 576).to(torch.bfloat16).cuda()
    before = pool.clone()
    src = torch.tensor([3, 300, 5], dtype=torch.int32, device="cuda")
    ip = torch.tensor([0, 3], dtype=torch.int32, device="cuda")
    dst = torch.tensor([254], dtype=torch.int64, device="cuda")   # third row would land at 256
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    va.verify_attn_defrag(pool, src, ip, dst, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == va.STATUS_BAD_SLOT | va.STATUS_BAD_DST
    assert torch.equal(pool[254], before[3])
    assert torch.equal(pool[:254], before[:254]) and torch.equal(pool[255], before[255])


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
def test_status_is_per_call_back_to_back(va, path):
    """The status word belongs to the last call: the split-K kernel may start
    while the tree-mask kernel (which clears the word) still runs, so every
    status write of the split-K kernel must come after it.  Calls go back to
    back on one stream, alternating inputs with and without bad slots, with no
    host synchronisation between them; the word is read after each pair and
    inside one captured graph."""
    s = synth.Spec("pc", B=1, H=8, T=16, prefix=[2000], num_slots=8192, seed=61)
    _need(va, path, s.B, s.T, s.H)
    w = synth.make(s)
    d_ok = _gpu.to_device(w)
    d_bad = dict(d_ok)
    bad = w.slot_idx.clone()
    bad[3] = 8192 + 11
    bad[1500] = -2
    d_bad["slot_idx"] = bad.cuda()
    ws, ns = va.alloc_workspace(s.B, s.T, s.H, 0, path)
    out = torch.empty(s.T, s.H, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(s.T, s.H, dtype=torch.float32, device="cuda")

    def call(dd):
        va.verify_attn_paged(dd["q"], dd["kv_pool"], dd["slot_idx"], dd["kv_indptr"],
                             dd["prefix_len"], dd["parents"], sm_scale=s.sm_scale, nsplit=ns,
                             flags=path, workspace=ws, out=out, lse=lse)

    for _ in range(10):
        call(d_bad)
        call(d_ok)
        assert va.read_status(ws) == 0
        call(d_ok)
        call(d_bad)
        assert va.read_status(ws) == va.STATUS_BAD_SLOT

    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        call(d_ok)
    torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    for first, second, want in ((d_bad, d_ok, 0), (d_ok, d_bad, va.STATUS_BAD_SLOT)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(first)
            call(second)
        for _ in range(5):
            g.replay()
            assert va.read_status(ws) == want
    ref_o, ref_l = _gpu.reference(w)
    call(d_ok)
    _gpu.compare(out, lse, ref_o, ref_l)


def test_prepared_call_relaunches_on_new_contents(va):
    """A call prepared once and launched again after new queries, slots and
    parents were copied into the same buffers computes the new step."""
    s1 = synth.Spec("prep1", B=2, H=8, T=8, prefix=[300, 120], num_slots=4096, seed=81)
    s2 = synth.Spec("prep2", B=2, H=8, T=8, prefix=[300, 120], num_slots=4096, seed=82)
    w1, w2 = synth.make(s1), synth.make(s2)
    d = _gpu.to_device(w1)
    kv2 = w2.kv_pool.cuda()
    call = va.prepare_paged(d["q"], kv2, d["slot_idx"], d["kv_indptr"], d["prefix_len"],
                            d["parents"], sm_scale=s1.sm_scale)
    out, lse = call()
    torch.cuda.synchronize()
    w1.kv_pool = w2.kv_pool          # both steps read the second pool
    ref_o, ref_l = _gpu.reference(w1)
    _gpu.compare(out, lse, ref_o, ref_l)
    d["q"].copy_(w2.q)
    d["slot_idx"].copy_(w2.slot_idx)
    d["parents"].copy_(w2.parents)
    out2, lse2 = call()
    torch.cuda.synchronize()
    assert out2.data_ptr() == out.data_ptr()
    ref_o, ref_l = _gpu.reference(w2)
    _gpu.compare(out2, lse2, ref_o, ref_l)


@pytest.mark.parametrize("path", list(PATHS.values()), ids=list(PATHS))
@pytest.mark.parametrize("scale", [0.0, -0.0721, 0.31])
def test_scale_sign(va, path, scale):
    """The tensor-core softmax keeps raw scores and scales their maximum when
    the scale is positive, and scales every score otherwise: both branches,
    and a scale of zero (every visible key weighs the same), against the
    oracle, with whole 64-key tiles and a ragged one."""
    s = synth.Spec("scale", B=2, H=8, T=16, prefix=[900, 131], num_slots=8192, seed=97,
                   sm_scale=scale)
    _need(va, path, s.B, s.T, s.H)
    w = synth.make(s)
    d = _gpu.to_device(w)
    out, lse = _gpu.run(va, d, w, path=path, nsplit=3)
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out, lse, ref_o, ref_l)


def test_many_small_requests(va):
    """300 requests of 0-200 prefix keys (H=4, T=4): a grid of 300 requests
    deep, a split count near 1 and the warp-per-row merge, every row against
    the oracle."""
    g = torch.Generator().manual_seed(123)
    pre = [int(x) for x in torch.randint(0, 201, (300,), generator=g)]
    s = synth.Spec("many", B=300, H=4, T=4, prefix=pre, num_slots=1 << 16, seed=124)
    w = synth.make(s)
    d = _gpu.to_device(w)
    ws, ns = va.alloc_workspace(s.B, s.T, s.H)
    out, lse = _gpu.run(va, d, w, nsplit=ns, workspace=ws)
    assert va.read_status(ws) == 0
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("H,T,prefix,layout", [
    (64, 16, [3000], "scattered"),
    (64, 16, [2000, 5001], "contiguous"),
    (24, 10, [1700], "scattered"),      # 240 rows: one unit, its second half partly padding
    (8, 32, [900, 40], "scattered"),    # 256 rows
])
def test_tensor_core_shapes_agree(va, H, T, prefix, layout):
    """Two-SM products (VA_PATH_TC at more than 128 rows) against one-SM
    products (VA_PATH_TC_1SM) at the same split count: the same per-row
    arithmetic in the same order, so the same bits; both also against the
    oracle."""
    s = synth.Spec("shapes", B=len(prefix), H=H, T=T, prefix=prefix, num_slots=1 << 15,
                   layout=layout, seed=H * 7 + T)
    w = synth.make(s)
    d = _gpu.to_device(w)
    o2, l2 = _gpu.run(va, d, w, path=PATHS["tc"], nsplit=5)
    o1, l1 = _gpu.run(va, d, w, path=PATHS["tc1sm"], nsplit=5)
    torch.cuda.synchronize()
    diff = (o2.float() - o1.float()).abs().max().item()
    assert torch.equal(o2, o1) and torch.equal(l2, l1), f"max |out diff| {diff}"
    ref_o, ref_l = _gpu.reference(w)
    _gpu.compare(o2, l2, ref_o, ref_l)
