"""Python binding of libverifyattn.so -- GB300 (sm_103a) MLA tree-verify attention.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/verify_attn.h``.  PyTorch
provides device memory and streams.  There is no CPU fallback: if the shared
library has not been built, :func:`load` raises.

Names follow the C ABI: ``verify_attn_paged``, ``verify_attn_contiguous``,
``verify_attn_defrag``, ``workspace_bytes``, ``auto_nsplit``, ``init``,
``read_status``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import _builder as _build_mod

D_QK = 576
D_V = 512
T_MAX = 64

VA_OK = 0
ERRORS = {-1: "VA_ERR_NULL", -2: "VA_ERR_SHAPE", -3: "VA_ERR_ALIGN", -4: "VA_ERR_WORKSPACE",
          -5: "VA_ERR_UNSUPPORTED", -6: "VA_ERR_LAUNCH", -7: "VA_ERR_CUDA"}
STATUS_BAD_SLOT = 0x1
STATUS_BAD_PARENT = 0x2
STATUS_BAD_INDPTR = 0x4
STATUS_TIMEOUT = 0x8
STATUS_BAD_DST = 0x10
STATUS_BAD_MASK = 0x20
PATH_AUTO, PATH_FMA, PATH_TC, PATH_TC_1SM = 0, 1, 2, 3

LIB_PATH = _build_mod.LIB


class VaError(RuntimeError):
    def __init__(self, func: str, code: int):
        self.code = code
        super().__init__(f"{func} returned {code} ({ERRORS.get(code, 'unknown')})")


_lib = None
_inited = set()


def build(force: bool = False) -> str:
    """Compile the CUDA sources into libverifyattn.so (nvcc, sm_103a)."""
    return _build_mod.build(force=force)


def load() -> ctypes.CDLL:
    """Load libverifyattn.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libverifyattn.so is not built ({LIB_PATH}); run "
                           "mla_speculative_decode_gb300.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.va_version.argtypes = []
    lib.va_version.restype = i32
    lib.va_init.argtypes = [i32]
    lib.va_init.restype = i32
    lib.va_auto_nsplit.argtypes = [i32, i32, i32, i32]
    lib.va_auto_nsplit.restype = i32
    lib.va_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.va_workspace_bytes.restype = sz
    lib.verify_attn_paged.argtypes = [P, P, i64, i64, P, P, P, P, P, i32, i32, i32, f32, i32, i32,
                                      P, sz, P, P, P]
    lib.verify_attn_paged.restype = i32
    lib.verify_attn_contiguous.argtypes = [P, P, i64, i64, P, P, P, P, i32, i32, i32, f32, i32, i32,
                                           P, sz, P, P, P]
    lib.verify_attn_contiguous.restype = i32
    lib.verify_attn_segmented.argtypes = [P, P, i64, i64, P, P, P, P, P, i64, P, P, i32, i32,
                                          i32, f32, i32, i32, P, sz, P, P, P]
    lib.verify_attn_segmented.restype = i32
    lib.va_tree_accept_workspace_bytes.argtypes = [i32, i32, i64]
    lib.va_tree_accept_workspace_bytes.restype = sz
    lib.va_tree_accept.argtypes = [P, P, i64, P, P, P, i32, i32, P, sz, P, P, P, P, P]
    lib.va_tree_accept.restype = i32
    lib.va_tree_build.argtypes = [P, P, i32, i32, i32, i32, P, i64, P, P, P, P, P, P, P]
    lib.va_tree_build.restype = i32
    lib.verify_attn_defrag.argtypes = [P, i64, i64, P, P, P, P, i32, i64, P, P]
    lib.verify_attn_defrag.restype = i32
    lib.va_kv_append_contiguous.argtypes = [P, i64, i64, P, P, P, P, i32, i32, P, P, P]
    lib.va_kv_append_contiguous.restype = i32
    lib.va_kv_compact_accepted.argtypes = [P, i64, i64, P, P, P, P, P, i32, i32, P, P]
    lib.va_kv_compact_accepted.restype = i32
    lib.verify_attn_paged_noalloc.argtypes = [P, P, i64, i64, P, P, P, P, P, i32, i32, i32, f32,
                                              i32, i32, P, P, P]
    lib.verify_attn_paged_noalloc.restype = i32
    lib.va_set_partial_events.argtypes = [P, P]
    lib.va_set_partial_events.restype = i32
    lib.va_read_status.argtypes = [P, P, P]
    lib.va_read_status.restype = i32
    _lib = lib
    return lib


def _check(func: str, rc: int) -> int:
    if rc < 0:
        raise VaError(func, rc)
    return rc


def init(device: Optional[int] = None) -> None:
    """va_init for `device` (default: torch's current device); idempotent."""
    if device is None:
        device = torch.cuda.current_device()
    if device in _inited:
        return
    _check("va_init", load().va_init(int(device)))
    _inited.add(device)


def workspace_bytes(B: int, T: int, H: int, nsplit: int) -> int:
    n = load().va_workspace_bytes(B, T, H, nsplit)
    if n == 0:
        raise VaError("va_workspace_bytes", -2)
    return n


def auto_nsplit(B: int, T: int, H: int, flags: int = PATH_AUTO) -> int:
    init()
    return _check("va_auto_nsplit", load().va_auto_nsplit(B, T, H, flags))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, name: str, dtype) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def alloc_workspace(B: int, T: int, H: int, nsplit: int = 0, flags: int = PATH_AUTO,
                    device=None) -> Tuple[torch.Tensor, int]:
    """A workspace tensor for these sizes and the nsplit it was sized for."""
    ns = nsplit if nsplit > 0 else auto_nsplit(B, T, H, flags)
    n = workspace_bytes(B, T, H, ns)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda"), ns


def _dims(q: torch.Tensor, B: int) -> Tuple[int, int]:
    """(T, H) of a query tensor [B*T, H, 576] for B requests.  The C ABI takes
    no tensor sizes, so a query block that does not split into B requests is
    rejected here, before any pointer reaches the library."""
    if q.dim() != 3 or q.shape[2] != D_QK:
        raise ValueError(f"q must be [B*T, H, {D_QK}], got {tuple(q.shape)}")
    if B < 1 or q.shape[0] % B != 0 or q.shape[0] == 0:
        raise ValueError(f"q has {q.shape[0]} rows, not a positive multiple of B={B}")
    return q.shape[0] // B, q.shape[1]


def _outputs(rows: int, H: int, device, out, lse):
    """Allocates out / lse when not given; a given one must have the step's
    exact shape (the kernels write [rows, H, 512] and [rows, H] through a bare
    pointer, so an undersized buffer would be written past its end)."""
    if out is None:
        out = torch.empty(rows, H, D_V, dtype=torch.bfloat16, device=device)
    if lse is None:
        lse = torch.empty(rows, H, dtype=torch.float32, device=device)
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    if tuple(out.shape) != (rows, H, D_V):
        raise ValueError(f"out must be [{rows}, {H}, {D_V}], got {tuple(out.shape)}")
    if tuple(lse.shape) != (rows, H):
        raise ValueError(f"lse must be [{rows}, {H}], got {tuple(lse.shape)}")
    return out, lse


def _tree_args(tree_parent, tree_bits, B: int, T: int):
    """Pointers of the tree arguments; the one used must hold B*T entries."""
    if tree_bits is not None:
        _dev(tree_bits, "tree_bits", torch.int64)
        if tree_bits.numel() != B * T:
            raise ValueError(f"tree_bits must hold B*T = {B * T} masks")
    elif tree_parent is not None:
        _dev(tree_parent, "tree_parent", torch.int32)
        if tree_parent.numel() != B * T:
            raise ValueError(f"tree_parent must hold B*T = {B * T} parents")
    return _ptr(tree_parent), _ptr(tree_bits)


class PreparedCall:
    """One verify call whose arguments were checked and marshalled once.

    Calling it launches the step again on the same buffers, whose contents may
    change between calls (new queries, slot tables, trees copied into them), on
    the stream it was prepared for: the host work per step is one C call.  The
    tensors it refers to must stay alive; `out` and `lse` are its outputs.
    """

    def __init__(self, name: str, args: tuple, out: torch.Tensor, lse: torch.Tensor, keep: tuple):
        self._fn = getattr(load(), name)
        self._name = name
        self._args = args
        self.out, self.lse = out, lse
        self._keep = keep          # the tensors behind the pointers

    def __call__(self) -> Tuple[torch.Tensor, torch.Tensor]:
        rc = self._fn(*self._args)
        if rc < 0:
            raise VaError(self._name, rc)
        return self.out, self.lse


def prepare_paged(q: torch.Tensor, kv_pool: torch.Tensor, slot_idx: torch.Tensor,
                  kv_indptr: torch.Tensor, prefix_len: torch.Tensor,
                  tree_parent: Optional[torch.Tensor] = None,
                  tree_bits: Optional[torch.Tensor] = None, *, sm_scale: float,
                  nsplit: int = 0, flags: int = PATH_AUTO,
                  workspace: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  stream=None) -> PreparedCall:
    """verify_attn_paged's checks and marshalling, done once: returns a
    PreparedCall that launches the step on these buffers each time it is called."""
    init(q.device.index)
    _dev(q, "q", torch.bfloat16)
    _dev(kv_pool, "kv_pool", torch.bfloat16)
    _dev(slot_idx, "slot_idx", torch.int32)
    _dev(kv_indptr, "kv_indptr", torch.int32)
    _dev(prefix_len, "prefix_len", torch.int32)
    if kv_pool.dim() != 2:
        raise ValueError("kv_pool must be [num_slots, stride]")
    B = prefix_len.shape[0]
    T, H = _dims(q, B)
    if workspace is None:
        workspace, nsplit = alloc_workspace(B, T, H, nsplit, flags, q.device)
    out, lse = _outputs(q.shape[0], H, q.device, out, lse)
    par, bits = _tree_args(tree_parent, tree_bits, B, T)
    args = (_ptr(q), _ptr(kv_pool), kv_pool.shape[0], kv_pool.stride(0), _ptr(slot_idx),
            _ptr(kv_indptr), _ptr(prefix_len), par, bits, B, T, H, float(sm_scale), nsplit, flags,
            _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse), _stream(stream))
    return PreparedCall("verify_attn_paged", args, out, lse,
                        (q, kv_pool, slot_idx, kv_indptr, prefix_len, tree_parent, tree_bits,
                         workspace))


def verify_attn_paged(q: torch.Tensor, kv_pool: torch.Tensor, slot_idx: torch.Tensor,
                      kv_indptr: torch.Tensor, prefix_len: torch.Tensor,
                      tree_parent: Optional[torch.Tensor] = None,
                      tree_bits: Optional[torch.Tensor] = None, *, sm_scale: float,
                      nsplit: int = 0, flags: int = PATH_AUTO,
                      workspace: Optional[torch.Tensor] = None,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Paged MLA tree-verify attention; returns (out bf16 [B*T, H, 512], lse fp32 [B*T, H]).

    q [B*T, H, 576] bf16; kv_pool [num_slots, stride] bf16; slot_idx int32;
    kv_indptr int32 [B+1]; prefix_len int32 [B]; tree_parent int32 [B, T] or
    tree_bits int64 [B, T] (bit patterns of uint64 masks).  All CUDA tensors.
    """
    return prepare_paged(q, kv_pool, slot_idx, kv_indptr, prefix_len, tree_parent, tree_bits,
                         sm_scale=sm_scale, nsplit=nsplit, flags=flags, workspace=workspace,
                         out=out, lse=lse, stream=stream)()


def verify_attn_contiguous(q: torch.Tensor, kv_pool: torch.Tensor, kv_start: torch.Tensor,
                           prefix_len: torch.Tensor, tree_parent: Optional[torch.Tensor] = None,
                           tree_bits: Optional[torch.Tensor] = None, *, sm_scale: float,
                           nsplit: int = 0, flags: int = PATH_AUTO,
                           workspace: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Contiguous-KV variant: request b's keys are pool rows kv_start[b] + j (int64 [B])."""
    init(q.device.index)
    _dev(q, "q", torch.bfloat16)
    _dev(kv_pool, "kv_pool", torch.bfloat16)
    _dev(kv_start, "kv_start", torch.int64)
    _dev(prefix_len, "prefix_len", torch.int32)
    if kv_pool.dim() != 2:
        raise ValueError("kv_pool must be [num_slots, stride]")
    B = prefix_len.shape[0]
    T, H = _dims(q, B)
    if workspace is None:
        workspace, nsplit = alloc_workspace(B, T, H, nsplit, flags, q.device)
    out, lse = _outputs(q.shape[0], H, q.device, out, lse)
    par, bits = _tree_args(tree_parent, tree_bits, B, T)
    rc = load().verify_attn_contiguous(
        _ptr(q), _ptr(kv_pool), kv_pool.shape[0], kv_pool.stride(0), _ptr(kv_start),
        _ptr(prefix_len), par, bits, B, T, H, float(sm_scale), nsplit, flags, _ptr(workspace),
        workspace.numel(), _ptr(out), _ptr(lse), _stream(stream))
    _check("verify_attn_contiguous", rc)
    return out, lse


def verify_attn_segmented(q: torch.Tensor, kv_pool: torch.Tensor, kv_indices: torch.Tensor,
                          kv_indptr: torch.Tensor, out_cache_loc: torch.Tensor,
                          custom_mask: Optional[torch.Tensor] = None,
                          draft_kv: Optional[torch.Tensor] = None,
                          tree_parent: Optional[torch.Tensor] = None,
                          tree_bits: Optional[torch.Tensor] = None, *, sm_scale: float,
                          nsplit: int = 0, flags: int = PATH_AUTO,
                          workspace: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Two-list variant: request b's prefix slots are kv_indices[kv_indptr[b]:kv_indptr[b+1]]
    (int32), its draft nodes' slots out_cache_loc[b*T:(b+1)*T] (int32 [B*T]); the tree is a
    dense extend mask (uint8 or bool, rows of prefix + T entries, only the last T read), or
    tree_parent / tree_bits as for verify_attn_paged.  With draft_kv (bf16 [B*T, 576]) the
    call first writes those rows into the pool at out_cache_loc."""
    init(q.device.index)
    _dev(q, "q", torch.bfloat16)
    _dev(kv_pool, "kv_pool", torch.bfloat16)
    _dev(kv_indices, "kv_indices", torch.int32)
    _dev(kv_indptr, "kv_indptr", torch.int32)
    _dev(out_cache_loc, "out_cache_loc", torch.int32)
    if kv_pool.dim() != 2:
        raise ValueError("kv_pool must be [num_slots, stride]")
    B = kv_indptr.shape[0] - 1
    T, H = _dims(q, B)
    if out_cache_loc.numel() != B * T:
        raise ValueError("out_cache_loc must hold B*T slots")
    mask_ptr, mask_len = None, 0
    if custom_mask is not None:
        if custom_mask.dtype == torch.bool:
            custom_mask = custom_mask.view(torch.uint8)
        _dev(custom_mask, "custom_mask", torch.uint8)
        mask_ptr, mask_len = _ptr(custom_mask), custom_mask.numel()
    if draft_kv is not None:
        _dev(draft_kv, "draft_kv", torch.bfloat16)
        if tuple(draft_kv.shape) != (B * T, D_QK):
            raise ValueError("draft_kv must be [B*T, 576]")
    if workspace is None:
        workspace, nsplit = alloc_workspace(B, T, H, nsplit, flags, q.device)
    out, lse = _outputs(q.shape[0], H, q.device, out, lse)
    par, bits = _tree_args(tree_parent, tree_bits, B, T)
    rc = load().verify_attn_segmented(
        _ptr(q), _ptr(kv_pool), kv_pool.shape[0], kv_pool.stride(0), _ptr(kv_indices),
        _ptr(kv_indptr), _ptr(out_cache_loc), _ptr(draft_kv), mask_ptr, mask_len, par, bits,
        B, T, H,
        float(sm_scale), nsplit, flags, _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
        _stream(stream))
    _check("verify_attn_segmented", rc)
    return out, lse


def verify_attn_defrag(kv_pool: torch.Tensor, src_slots: torch.Tensor, src_indptr: torch.Tensor,
                       dst_base: torch.Tensor, slot_idx_out: Optional[torch.Tensor] = None,
                       max_rows: Optional[int] = None, status: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """Copy request b's rows src_slots[indptr[b]:indptr[b+1]] to dst_base[b] + i (in place)."""
    init(kv_pool.device.index)
    _dev(kv_pool, "kv_pool", torch.bfloat16)
    _dev(src_slots, "src_slots", torch.int32)
    _dev(src_indptr, "src_indptr", torch.int32)
    _dev(dst_base, "dst_base", torch.int64)
    if slot_idx_out is not None:
        _dev(slot_idx_out, "slot_idx_out", torch.int32)
    if status is not None:
        _dev(status, "status", torch.int32)
    B = dst_base.shape[0]
    rows = int(max_rows) if max_rows is not None else max(1, src_slots.numel())
    rc = load().verify_attn_defrag(
        _ptr(kv_pool), kv_pool.shape[0], kv_pool.stride(0), _ptr(src_slots), _ptr(src_indptr),
        _ptr(dst_base), _ptr(slot_idx_out), B, rows, _ptr(status), _stream(stream))
    _check("verify_attn_defrag", rc)


def _placement_args(kv_pool, kv_start, prefix_len, kv_capacity):
    _dev(kv_pool, "kv_pool", torch.bfloat16)
    _dev(kv_start, "kv_start", torch.int64)
    _dev(prefix_len, "prefix_len", torch.int32)
    _dev(kv_capacity, "kv_capacity", torch.int32)
    B = kv_start.numel()
    if prefix_len.numel() != B or kv_capacity.numel() != B:
        raise ValueError("kv_start, prefix_len and kv_capacity need one entry per request")
    if kv_pool.dim() != 2 or kv_pool.stride(1) != 1:
        raise ValueError("kv_pool must be a row-major [num_slots, stride] tensor")
    return B


def kv_append_contiguous(kv_pool: torch.Tensor, kv_start: torch.Tensor, prefix_len: torch.Tensor,
                         kv_capacity: torch.Tensor, draft_kv: torch.Tensor,
                         out_cache_loc: Optional[torch.Tensor] = None,
                         status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Draft latents of request b (draft_kv rows b*T .. b*T+T-1) into the rows
    right after its prefix, kv_start[b] + prefix_len[b] + i, within its
    reserved kv_capacity[b] rows (see va_kv_append_contiguous in
    verify_attn.h); out_cache_loc (int32 [B*T]) receives the rows."""
    init(kv_pool.device.index)
    B = _placement_args(kv_pool, kv_start, prefix_len, kv_capacity)
    _dev(draft_kv, "draft_kv", torch.bfloat16)
    if draft_kv.dim() != 2 or draft_kv.shape[1] != D_QK or draft_kv.shape[0] % B != 0 \
            or not draft_kv.is_contiguous():
        raise ValueError("draft_kv must be a contiguous [B*T, 576] tensor")
    T = draft_kv.shape[0] // B
    if out_cache_loc is not None:
        _dev(out_cache_loc, "out_cache_loc", torch.int32)
        if out_cache_loc.numel() != B * T:
            raise ValueError("out_cache_loc needs B*T entries")
    if status is not None:
        _dev(status, "status", torch.int32)
    rc = load().va_kv_append_contiguous(
        _ptr(kv_pool), kv_pool.shape[0], kv_pool.stride(0), _ptr(kv_start), _ptr(prefix_len),
        _ptr(kv_capacity), _ptr(draft_kv), B, T, _ptr(out_cache_loc), _ptr(status),
        _stream(stream))
    _check("va_kv_append_contiguous", rc)


def kv_compact_accepted(kv_pool: torch.Tensor, kv_start: torch.Tensor, prefix_len: torch.Tensor,
                        kv_capacity: torch.Tensor, accept_len: torch.Tensor,
                        accept_nodes: torch.Tensor, status: Optional[torch.Tensor] = None,
                        stream=None) -> None:
    """The accepted path of request b (accept_nodes[b, :accept_len[b]]) moved
    to the rows right after its prefix, and prefix_len[b] advanced by
    accept_len[b], in place on the device (see va_kv_compact_accepted in
    verify_attn.h)."""
    init(kv_pool.device.index)
    B = _placement_args(kv_pool, kv_start, prefix_len, kv_capacity)
    _dev(accept_len, "accept_len", torch.int32)
    _dev(accept_nodes, "accept_nodes", torch.int32)
    if accept_len.numel() != B or accept_nodes.numel() % B != 0:
        raise ValueError("accept_len needs B entries and accept_nodes B*T")
    T = accept_nodes.numel() // B
    if status is not None:
        _dev(status, "status", torch.int32)
    rc = load().va_kv_compact_accepted(
        _ptr(kv_pool), kv_pool.shape[0], kv_pool.stride(0), _ptr(kv_start), _ptr(prefix_len),
        _ptr(kv_capacity), _ptr(accept_len), _ptr(accept_nodes), B, T, _ptr(status),
        _stream(stream))
    _check("va_kv_compact_accepted", rc)


def tree_accept(root_logits: torch.Tensor, logits: torch.Tensor, draft_tokens: torch.Tensor,
                tree_parent: torch.Tensor, draft_slots: Optional[torch.Tensor] = None, *,
                workspace: Optional[torch.Tensor] = None, outputs=None, stream=None):
    """Greedy tree acceptance after verify.

    root_logits fp32 [B, V] (the target's logits at the last prefix position),
    logits fp32 [B, T, V] (at each draft node), draft_tokens int32 [B, T],
    tree_parent int32 [B, T], draft_slots int32 [B, T] or None.  Returns
    (accept_len int32 [B], accept_nodes int32 [B, T], accept_slots int32 [B, T],
    bonus_token int32 [B], workspace); see va_tree_accept in verify_attn.h.
    `outputs` = (accept_len, accept_nodes, accept_slots, bonus_token) tensors to
    write into instead of new ones.
    """
    init(logits.device.index)
    _dev(root_logits, "root_logits", torch.float32)
    _dev(logits, "logits", torch.float32)
    _dev(draft_tokens, "draft_tokens", torch.int32)
    _dev(tree_parent, "tree_parent", torch.int32)
    if draft_slots is not None:
        _dev(draft_slots, "draft_slots", torch.int32)
    if logits.dim() != 3:
        raise ValueError("logits must be [B, T, V]")
    B, T, V = logits.shape
    if workspace is None:
        n = load().va_tree_accept_workspace_bytes(B, T, V)
        if n == 0:
            raise VaError("va_tree_accept_workspace_bytes", -2)
        workspace = torch.empty(n, dtype=torch.uint8, device=logits.device)
    dev = logits.device
    if outputs is None:
        outputs = (torch.empty(B, dtype=torch.int32, device=dev),
                   torch.empty(B, T, dtype=torch.int32, device=dev),
                   torch.empty(B, T, dtype=torch.int32, device=dev),
                   torch.empty(B, dtype=torch.int32, device=dev))
    alen, nodes, slots, bonus = outputs
    for t, name in zip(outputs, ("accept_len", "accept_nodes", "accept_slots", "bonus_token")):
        _dev(t, name, torch.int32)
    rc = load().va_tree_accept(_ptr(root_logits), _ptr(logits), V, _ptr(draft_tokens),
                               _ptr(tree_parent), _ptr(draft_slots), B, T, _ptr(workspace),
                               workspace.numel(), _ptr(alen), _ptr(nodes), _ptr(slots),
                               _ptr(bonus), _stream(stream))
    _check("va_tree_accept", rc)
    return alen, nodes, slots, bonus, workspace


TREE_MAX_DEPTH = 15
TREE_MAX_CAND = 16


def tree_build(cand_tokens: torch.Tensor, cand_logp: torch.Tensor, T: int,
               free_slots: Optional[torch.Tensor] = None,
               free_head: Optional[torch.Tensor] = None, *, outputs=None,
               status: Optional[torch.Tensor] = None, stream=None):
    """Draft tree of each request from the drafter's candidates, on the device.

    cand_tokens int32 [B, D, K], cand_logp fp32 [B, D, K]: K candidate tokens
    with log-probabilities per draft position.  The tree is grown best first
    (see va_tree_build in verify_attn.h).  With free_slots (int32) and
    free_head (int32 [1], device), node i of request b takes the pool slot
    free_slots[head + b*T + i] and the head advances by B*T.  Returns
    (tree_parent int32 [B, T], draft_tokens int32 [B, T], node_depth int32
    [B, T], out_cache_loc int32 [B*T] or None).  `outputs` = those tensors to
    write into instead of new ones.
    """
    init(cand_logp.device.index)
    _dev(cand_tokens, "cand_tokens", torch.int32)
    _dev(cand_logp, "cand_logp", torch.float32)
    if cand_tokens.dim() != 3 or tuple(cand_tokens.shape) != tuple(cand_logp.shape):
        raise ValueError("cand_tokens and cand_logp must both be [B, D, K]")
    B, D, K = cand_tokens.shape
    dev = cand_logp.device
    if (free_slots is None) != (free_head is None):
        raise ValueError("free_slots and free_head go together")
    if free_slots is not None:
        _dev(free_slots, "free_slots", torch.int32)
        _dev(free_head, "free_head", torch.int32)
        if free_head.numel() != 1:
            raise ValueError("free_head must hold one int32")
    if outputs is None:
        outputs = (torch.empty(B, T, dtype=torch.int32, device=dev),
                   torch.empty(B, T, dtype=torch.int32, device=dev),
                   torch.empty(B, T, dtype=torch.int32, device=dev),
                   torch.empty(B * T, dtype=torch.int32, device=dev)
                   if free_slots is not None else None)
    par, tok, depth, loc = outputs
    for t, n, size in ((par, "tree_parent", B * T), (tok, "draft_tokens", B * T),
                       (depth, "node_depth", B * T), (loc, "out_cache_loc", B * T)):
        if t is not None:
            _dev(t, n, torch.int32)
            if t.numel() != size:
                raise ValueError(f"{n} must hold {size} entries")
    if free_slots is not None and loc is None:
        raise ValueError("out_cache_loc is needed with free_slots")
    if status is not None:
        _dev(status, "status", torch.int32)
    rc = load().va_tree_build(_ptr(cand_tokens), _ptr(cand_logp), B, D, K, int(T),
                              _ptr(free_slots), 0 if free_slots is None else free_slots.numel(),
                              _ptr(free_head), _ptr(par), _ptr(tok), _ptr(depth),
                              _ptr(loc) if free_slots is not None else None, _ptr(status),
                              _stream(stream))
    _check("va_tree_build", rc)
    return par, tok, depth, (loc if free_slots is not None else None)


def read_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the workspace status word."""
    v = ctypes.c_uint32(0)
    _check("va_read_status", load().va_read_status(_ptr(workspace), ctypes.byref(v),
                                                   _stream(stream)))
    return int(v.value)


def set_partial_events(before=None, after=None) -> None:
    """Record torch.cuda.Event `before`/`after` around the split-K partial kernel
    of every following verify call (None, None stops)."""
    if before is None or after is None:
        load().va_set_partial_events(None, None)
        return
    for e in (before, after):
        if e.cuda_event == 0:
            e.record()          # the handle is created on first record
    load().va_set_partial_events(before.cuda_event, after.cuda_event)


NOALLOC_SCRATCH_BYTES = 16 << 20


def verify_attn_paged_noalloc(q: torch.Tensor, kv_pool: torch.Tensor, slot_idx: torch.Tensor,
                              kv_indptr: torch.Tensor, prefix_len: torch.Tensor,
                              tree_parent: Optional[torch.Tensor] = None,
                              tree_bits: Optional[torch.Tensor] = None, *, sm_scale: float,
                              nsplit: int = 0, flags: int = PATH_AUTO, out: torch.Tensor,
                              lse: torch.Tensor, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """verify_attn_paged without a workspace: the library's fixed scratch array is
    used instead, so nothing is allocated.  `out` and `lse` must be given."""
    init(q.device.index)
    for t, n, dt in ((q, "q", torch.bfloat16), (kv_pool, "kv_pool", torch.bfloat16),
                     (slot_idx, "slot_idx", torch.int32), (kv_indptr, "kv_indptr", torch.int32),
                     (prefix_len, "prefix_len", torch.int32), (out, "out", torch.bfloat16),
                     (lse, "lse", torch.float32)):
        _dev(t, n, dt)
    if kv_pool.dim() != 2:
        raise ValueError("kv_pool must be [num_slots, stride]")
    B = prefix_len.shape[0]
    T, H = _dims(q, B)
    _outputs(q.shape[0], H, q.device, out, lse)
    par, bits = _tree_args(tree_parent, tree_bits, B, T)
    rc = load().verify_attn_paged_noalloc(
        _ptr(q), _ptr(kv_pool), kv_pool.shape[0], kv_pool.stride(0), _ptr(slot_idx),
        _ptr(kv_indptr), _ptr(prefix_len), par, bits, B, T, H, float(sm_scale), nsplit, flags,
        _ptr(out), _ptr(lse), _stream(stream))
    _check("verify_attn_paged_noalloc", rc)
    return out, lse
