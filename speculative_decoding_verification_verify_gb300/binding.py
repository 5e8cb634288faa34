"""ctypes binding of libspecverify.so with the same entry-point names as include/spec_verify.h.

Argument marshalling only: tensors are checked and their device pointers handed to the C ABI
on the current CUDA stream; every step of verification runs in the library's CUDA kernels.
PyTorch supplies device memory (outputs, the workspace) and the stream.  There is no CPU
fallback: if the library is not built or no GPU is present, these functions raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import NamedTuple, Optional

import torch

from . import _build

BF16, FP32 = 0, 1
MODE_GREEDY, MODE_REJECTION, MODE_TREE, MODE_BLOCK = 0, 1, 2, 3
OK, EINVAL, EWORKSPACE, ECUDA, ETOOBIG = 0, -1, -2, -3, -4
NOALLOC_SCRATCH_BYTES = 4 << 20
DEV_OK, DEV_BAD_TOKEN, DEV_BAD_ROW, DEV_BAD_TREE, DEV_DUP_SIBLING = 0, 1, 2, 3, 4
DEV_BAD_KV_POSITION, DEV_BAD_KV_SLOT = 5, 6

_lib = None
_lock = threading.Lock()


class Options(ctypes.Structure):
    """spec_verify_options: a temperature per request (device float32 [B], 0 = greedy) or one
    temperature for all, and the relaxed thresholds of target-only decisions (1 = exact)."""
    _fields_ = [("temperatures", ctypes.c_void_p), ("temperature", ctypes.c_float),
                ("threshold_single", ctypes.c_float), ("threshold_acc", ctypes.c_float),
                ("top_k", ctypes.c_void_p), ("top_p", ctypes.c_void_p)]


def library_path() -> str:
    return _build.LIB_PATH


def _declare(lib):
    """Argument and result types of every entry point of include/spec_verify.h."""
    vp, i32, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float,
                             ctypes.c_size_t)
    lib.spec_verify_greedy.argtypes = [vp, i32, vp, i32, i32, i32, vp, vp, vp, sz, vp, vp]
    lib.spec_verify_greedy.restype = i32
    lib.spec_verify_rejection.argtypes = [vp, i32, vp, vp, i32, i32, i32, f32, u64, u64, vp,
                                          vp, vp, vp, sz, vp, vp]
    lib.spec_verify_rejection.restype = i32
    lib.spec_verify_block.argtypes = [vp, i32, vp, vp, i32, i32, i32, f32, u64, u64, vp, vp,
                                      vp, sz, vp, vp]
    lib.spec_verify_block.restype = i32
    lib.spec_verify_tree.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, f32, u64, u64, vp,
                                     vp, vp, vp, sz, vp, vp]
    lib.spec_verify_tree.restype = i32
    lib.spec_verify_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.spec_verify_workspace_bytes.restype = sz
    lib.spec_verify_strerror.argtypes = [i32]
    lib.spec_verify_strerror.restype = ctypes.c_char_p
    lib.spec_verify_philox.argtypes = [u64, u64, i32, i32, vp, vp]
    lib.spec_verify_philox.restype = i32
    lib.spec_verify_rejection_noalloc.argtypes = [vp, i32, vp, vp, i32, i32, i32, f32, u64,
                                                  u64, vp, vp, vp, vp, vp]
    lib.spec_verify_rejection_noalloc.restype = i32
    lib.spec_verify_kv_compact.argtypes = [vp, ctypes.c_int64, sz, i32, sz, vp, i32, vp, vp,
                                           vp, vp, i32, i32, vp, vp]
    lib.spec_verify_kv_compact.restype = i32
    OP = ctypes.POINTER(Options)
    lib.spec_verify_rejection_ex.argtypes = [vp, i32, vp, vp, i32, i32, i32, OP, u64, u64, vp,
                                             vp, vp, vp, sz, vp, vp]
    lib.spec_verify_rejection_ex.restype = i32
    lib.spec_verify_tree_ex.argtypes = [vp, i32, vp, vp, i32, i32, i32, OP, u64, u64, vp, vp,
                                        vp, vp, sz, vp, vp]
    lib.spec_verify_tree_ex.restype = i32
    lib.spec_verify_plan_budget.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.spec_verify_plan_budget.restype = i32
    lib.spec_verify_plan_budget_workspace_bytes.argtypes = [i32, i32]
    lib.spec_verify_plan_budget_workspace_bytes.restype = sz
    lib.spec_verify_debug_fault.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    lib.spec_verify_debug_fault.restype = i32
    lib.spec_verify_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    lib.spec_verify_wait_timeouts.restype = i32
    return lib


def load_library():
    """Load libspecverify.so (in-tree).  Raises when it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with __graft_entry__.build() (nvcc, sm_103a)")
        _lib = _declare(ctypes.CDLL(path))
        return _lib


def load_debug_library():
    """The range-checked build (libspecverify_debug.so, compiled on first use): the same entry
    points, every kernel's global-memory indices checked (spec_verify_debug_fault reports)."""
    return _declare(ctypes.CDLL(_build.build_debug()))


@contextlib.contextmanager
def using_library(lib):
    """Route this module's wrappers through another build of the library (e.g. the debug one)."""
    global _lib
    load_library()
    with _lock:
        prev, _lib = _lib, lib
    try:
        yield lib
    finally:
        with _lock:
            _lib = prev


def spec_verify_debug_fault(lib=None) -> int:
    """The first out-of-range index recorded by a debug build since the last read (0: none)."""
    lib = lib or load_library()
    w = ctypes.c_uint64(0)
    rc = lib.spec_verify_debug_fault(ctypes.byref(w))
    if rc != OK:
        raise SpecVerifyError("spec_verify_debug_fault", rc)
    return int(w.value)


def spec_verify_wait_timeouts(lib=None) -> int:
    """Waits of the top-k / top-p ring kernel that ran out of time since the last read (0 in
    normal operation; their rows were finished by the general threshold kernel)."""
    lib = lib or load_library()
    n = ctypes.c_uint64(0)
    rc = lib.spec_verify_wait_timeouts(ctypes.byref(n))
    if rc != OK:
        raise SpecVerifyError("spec_verify_wait_timeouts", rc)
    return int(n.value)


def spec_verify_strerror(code: int) -> str:
    return load_library().spec_verify_strerror(int(code)).decode()


def spec_verify_workspace_bytes(mode: int, B: int, k_or_N: int, V: int) -> int:
    return int(load_library().spec_verify_workspace_bytes(mode, B, k_or_N, V))


class SpecVerifyError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code}: {spec_verify_strerror(code)}")
        self.code = code


# --------------------------------------------------------------------------------------------
# Marshalling helpers
# --------------------------------------------------------------------------------------------
_ws_cache: dict = {}
_plan_ws_cache: dict = {}


def workspace_for(nbytes: int, device: torch.device, stream: torch.cuda.Stream) -> torch.Tensor:
    """A zero-filled uint8 device buffer of at least nbytes, kept per (device, stream).

    The library leaves a workspace's counters zero after each call, so one zero-fill suffices.
    """
    key = (device.index, stream.cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _logits_dtype(logits: torch.Tensor) -> int:
    if logits.dtype == torch.bfloat16:
        return BF16
    if logits.dtype == torch.float32:
        return FP32
    raise TypeError(f"logits must be bfloat16 or float32, got {logits.dtype}")


def _check_dev(name: str, t: torch.Tensor, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _ws_and_status(nbytes, device, stream, workspace, dev_status):
    if workspace is None:
        workspace = workspace_for(nbytes, device, stream)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=device)
    return workspace, dev_status


class Result(NamedTuple):
    out_tokens: torch.Tensor
    accept_len: torch.Tensor
    dev_status: torch.Tensor
    accept_index: Optional[torch.Tensor] = None
    out_probs: Optional[torch.Tensor] = None


# --------------------------------------------------------------------------------------------
# Entry points
# --------------------------------------------------------------------------------------------
def spec_verify_greedy(logits: torch.Tensor, draft_ids: torch.Tensor, *, out_tokens=None,
                       accept_len=None, workspace=None, dev_status=None, stream=None) -> Result:
    """logits [B, k+1, V] (bf16 / fp32), draft_ids [B, k] int32 -> Result."""
    lib = load_library()
    _check_dev("logits", logits)
    B, k1, V = logits.shape
    k = k1 - 1
    _check_dev("draft_ids", draft_ids, torch.int32)
    if tuple(draft_ids.shape) != (B, k):
        raise ValueError("draft_ids must be [B, k]")
    dev = logits.device
    stream = stream or torch.cuda.current_stream(dev)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, k1), dtype=torch.int32, device=dev)
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = spec_verify_workspace_bytes(MODE_GREEDY, B, k, V)
    workspace, dev_status = _ws_and_status(nbytes, dev, stream, workspace, dev_status)
    rc = lib.spec_verify_greedy(_ptr(logits), _logits_dtype(logits), _ptr(draft_ids), B, k, V,
                                _ptr(out_tokens), _ptr(accept_len), _ptr(workspace),
                                workspace.numel(), _ptr(dev_status),
                                ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_greedy", rc)
    return Result(out_tokens, accept_len, dev_status)


def spec_verify_rejection(logits: torch.Tensor, draft_ids: torch.Tensor,
                          draft_probs: Optional[torch.Tensor] = None, *, temperature: float,
                          seed: int, offset: int, out_tokens=None, accept_len=None,
                          out_probs=None, want_probs: bool = False, workspace=None,
                          dev_status=None, stream=None) -> Result:
    """Standard rejection (draft_probs [B, k, V] fp32) or one-hot (draft_probs None)."""
    lib = load_library()
    _check_dev("logits", logits)
    B, k1, V = logits.shape
    k = k1 - 1
    _check_dev("draft_ids", draft_ids, torch.int32)
    if tuple(draft_ids.shape) != (B, k):
        raise ValueError("draft_ids must be [B, k]")
    if draft_probs is not None:
        _check_dev("draft_probs", draft_probs, torch.float32)
        if tuple(draft_probs.shape) != (B, k, V):
            raise ValueError("draft_probs must be [B, k, V]")
    dev = logits.device
    stream = stream or torch.cuda.current_stream(dev)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, k1), dtype=torch.int32, device=dev)
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    if out_probs is None and want_probs:
        out_probs = torch.empty((B, k1, 3), dtype=torch.float32, device=dev)
    nbytes = spec_verify_workspace_bytes(MODE_REJECTION, B, k, V)
    workspace, dev_status = _ws_and_status(nbytes, dev, stream, workspace, dev_status)
    rc = lib.spec_verify_rejection(_ptr(logits), _logits_dtype(logits), _ptr(draft_ids),
                                   _ptr(draft_probs), B, k, V, float(temperature),
                                   int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                   _ptr(out_tokens), _ptr(accept_len), _ptr(out_probs),
                                   _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                   ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_rejection", rc)
    return Result(out_tokens, accept_len, dev_status, None, out_probs)


def spec_verify_block(logits: torch.Tensor, draft_ids: torch.Tensor,
                      draft_probs: Optional[torch.Tensor] = None, *, temperature: float,
                      seed: int, offset: int, out_tokens=None, accept_len=None, workspace=None,
                      dev_status=None, stream=None) -> Result:
    """Block verification of a chain: draft_probs [B, k, V] fp32, or None for one-hot drafts."""
    lib = load_library()
    _check_dev("logits", logits)
    B, k1, V = logits.shape
    k = k1 - 1
    _check_dev("draft_ids", draft_ids, torch.int32)
    if tuple(draft_ids.shape) != (B, k):
        raise ValueError("draft_ids must be [B, k]")
    if draft_probs is not None:
        _check_dev("draft_probs", draft_probs, torch.float32)
        if tuple(draft_probs.shape) != (B, k, V):
            raise ValueError("draft_probs must be [B, k, V]")
    dev = logits.device
    stream = stream or torch.cuda.current_stream(dev)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, k1), dtype=torch.int32, device=dev)
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = spec_verify_workspace_bytes(MODE_BLOCK, B, k, V)
    workspace, dev_status = _ws_and_status(nbytes, dev, stream, workspace, dev_status)
    rc = lib.spec_verify_block(_ptr(logits), _logits_dtype(logits), _ptr(draft_ids), _ptr(draft_probs),
                               B, k, V, float(temperature), int(seed) & (2**64 - 1),
                               int(offset) & (2**64 - 1), _ptr(out_tokens), _ptr(accept_len),
                               _ptr(workspace), workspace.numel(), _ptr(dev_status),
                               ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_block", rc)
    return Result(out_tokens, accept_len, dev_status)


def spec_verify_tree(logits: torch.Tensor, node_tokens: torch.Tensor, parents: torch.Tensor, *,
                     mode: int, temperature: float = 1.0, seed: int = 0, offset: int = 0,
                     out_tokens=None, accept_index=None, accept_len=None, workspace=None,
                     dev_status=None, stream=None) -> Result:
    """logits [B, N, V]; node_tokens, parents [B, N] int32; mode 0 greedy, 1 target-only."""
    lib = load_library()
    _check_dev("logits", logits)
    B, N, V = logits.shape
    _check_dev("node_tokens", node_tokens, torch.int32)
    _check_dev("parents", parents, torch.int32)
    if tuple(node_tokens.shape) != (B, N) or tuple(parents.shape) != (B, N):
        raise ValueError("node_tokens and parents must be [B, N]")
    dev = logits.device
    stream = stream or torch.cuda.current_stream(dev)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, N), dtype=torch.int32, device=dev)
    accept_index = accept_index if accept_index is not None else torch.empty((B, N), dtype=torch.int32, device=dev)
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = spec_verify_workspace_bytes(MODE_TREE, B, N, V)
    workspace, dev_status = _ws_and_status(nbytes, dev, stream, workspace, dev_status)
    rc = lib.spec_verify_tree(_ptr(logits), _logits_dtype(logits), _ptr(node_tokens),
                              _ptr(parents), B, N, V, int(mode), float(temperature),
                              int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                              _ptr(out_tokens), _ptr(accept_index), _ptr(accept_len),
                              _ptr(workspace), workspace.numel(), _ptr(dev_status),
                              ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_tree", rc)
    return Result(out_tokens, accept_len, dev_status, accept_index)


def spec_verify_philox(seed: int, offset: int, n_slot: int, n_req: int, out=None,
                       device=None, stream=None) -> torch.Tensor:
    """Raw Philox4x32-10 words [n_slot, n_req, 4] (as int32 bit patterns) for the library's
    counter layout (slot, request, offset)."""
    lib = load_library()
    device = torch.device(device or "cuda")
    stream = stream or torch.cuda.current_stream(device)
    if out is None:
        out = torch.empty((n_slot, n_req, 4), dtype=torch.int32, device=device)
    rc = lib.spec_verify_philox(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), n_slot, n_req,
                                _ptr(out), ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_philox", rc)
    return out


def spec_verify_rejection_noalloc(logits: torch.Tensor, draft_ids: torch.Tensor,
                                  draft_probs: Optional[torch.Tensor] = None, *, temperature: float,
                                  seed: int, offset: int, out_tokens: torch.Tensor,
                                  accept_len: torch.Tensor, out_probs=None, dev_status=None,
                                  stream=None) -> Result:
    """spec_verify_rejection without a workspace, for callers that cannot allocate device memory
    while they verify: the library's built-in scratch is used instead.  The caller passes every
    output buffer (and dev_status, or None), so this wrapper allocates nothing either."""
    lib = load_library()
    _check_dev("logits", logits)
    B, k1, V = logits.shape
    k = k1 - 1
    _check_dev("draft_ids", draft_ids, torch.int32)
    if draft_probs is not None:
        _check_dev("draft_probs", draft_probs, torch.float32)
    _check_dev("out_tokens", out_tokens, torch.int32)
    _check_dev("accept_len", accept_len, torch.int32)
    stream = stream or torch.cuda.current_stream(logits.device)
    rc = lib.spec_verify_rejection_noalloc(_ptr(logits), _logits_dtype(logits), _ptr(draft_ids),
                                           _ptr(draft_probs), B, k, V, float(temperature),
                                           int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                           _ptr(out_tokens), _ptr(accept_len), _ptr(out_probs),
                                           _ptr(dev_status), ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_rejection_noalloc", rc)
    return Result(out_tokens, accept_len, dev_status, None, out_probs)


def spec_verify_kv_compact(kv_pool: torch.Tensor, slot_table: torch.Tensor,
                           committed: torch.Tensor, accept_index: torch.Tensor,
                           accept_len: torch.Tensor, *, stacked: bool = False, committed_out=None,
                           dev_status=None, stream=None):
    """Move each request's accepted-path KV rows (as spec_verify_tree reports them) to the
    positions right after its committed prefix, in place in kv_pool, and return
    (committed_out, dev_status).

    kv_pool is [num_slots, ...] with contiguous slot rows, or with stacked=True
    [planes, num_slots, ...] (one plane per layer and K or V) where each plane is contiguous and
    planes may be any 16-byte multiple apart; a slot row's bytes must be a multiple of 16.
    slot_table [B, max_pos], committed [B], accept_index [B, N] and accept_len [B] are int32
    CUDA tensors."""
    lib = load_library()
    if not kv_pool.is_cuda:
        raise ValueError("kv_pool must be a CUDA tensor")
    for name, t in (("slot_table", slot_table), ("committed", committed),
                    ("accept_index", accept_index), ("accept_len", accept_len)):
        _check_dev(name, t, torch.int32)
    B, N = accept_index.shape
    if slot_table.dim() != 2 or slot_table.shape[0] != B or tuple(committed.shape) != (B,) \
            or tuple(accept_len.shape) != (B,):
        raise ValueError("slot_table must be [B, max_pos], committed and accept_len [B]")
    if stacked:
        if kv_pool.dim() < 3 or not kv_pool[0].is_contiguous():
            raise ValueError("a stacked kv_pool is [planes, num_slots, ...] with contiguous planes")
        planes, num_slots = kv_pool.shape[0], kv_pool.shape[1]
        row_bytes = kv_pool[0, 0].numel() * kv_pool.element_size()
        plane_stride = kv_pool.stride(0) * kv_pool.element_size()
    else:
        if kv_pool.dim() < 2 or not kv_pool.is_contiguous():
            raise ValueError("kv_pool must be a contiguous [num_slots, ...] tensor")
        planes, num_slots = 1, kv_pool.shape[0]
        row_bytes = kv_pool[0].numel() * kv_pool.element_size()
        plane_stride = 0
    dev = kv_pool.device
    stream = stream or torch.cuda.current_stream(dev)
    if committed_out is None:
        committed_out = torch.empty(B, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.spec_verify_kv_compact(_ptr(kv_pool), int(num_slots), int(row_bytes), int(planes),
                                    int(plane_stride), _ptr(slot_table), slot_table.shape[1],
                                    _ptr(committed), _ptr(committed_out), _ptr(accept_index),
                                    _ptr(accept_len), B, N, _ptr(dev_status),
                                    ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_kv_compact", rc)
    return committed_out, dev_status


def _options(temperatures, temperature, threshold_single, threshold_acc, B, device, top_k=None,
             top_p=None):
    for name, t, dt in (("temperatures", temperatures, torch.float32), ("top_k", top_k, torch.int32),
                        ("top_p", top_p, torch.float32)):
        if t is not None:
            _check_dev(name, t, dt)
            if tuple(t.shape) != (B,) or t.device != device:
                raise ValueError(f"{name} must be a [B] {dt} tensor on the logits' device")
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return Options(ptr(temperatures), float(temperature), float(threshold_single), float(threshold_acc),
                   ptr(top_k), ptr(top_p))


def spec_verify_rejection_ex(logits: torch.Tensor, draft_ids: torch.Tensor,
                             draft_probs: Optional[torch.Tensor] = None, *, temperatures=None,
                             temperature: float = 1.0, threshold_single: float = 1.0,
                             threshold_acc: float = 1.0, top_k=None, top_p=None, seed: int = 0,
                             offset: int = 0,
                             out_tokens=None, accept_len=None, out_probs=None, workspace=None,
                             dev_status=None, stream=None) -> Result:
    """spec_verify_rejection with a temperature per request (temperatures [B], 0 = greedy
    request), relaxed thresholds for target-only decisions, and per-request top-k / top-p
    (top_k [B] int32, top_p [B] float32) on the target distribution."""
    lib = load_library()
    _check_dev("logits", logits)
    B, k1, V = logits.shape
    k = k1 - 1
    _check_dev("draft_ids", draft_ids, torch.int32)
    if draft_probs is not None:
        _check_dev("draft_probs", draft_probs, torch.float32)
    dev = logits.device
    stream = stream or torch.cuda.current_stream(dev)
    opt = _options(temperatures, temperature, threshold_single, threshold_acc, B, dev, top_k, top_p)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, k1), dtype=torch.int32, device=dev)
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = spec_verify_workspace_bytes(MODE_REJECTION, B, k, V)
    workspace, dev_status = _ws_and_status(nbytes, dev, stream, workspace, dev_status)
    rc = lib.spec_verify_rejection_ex(_ptr(logits), _logits_dtype(logits), _ptr(draft_ids),
                                      _ptr(draft_probs), B, k, V, ctypes.byref(opt),
                                      int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                      _ptr(out_tokens), _ptr(accept_len), _ptr(out_probs),
                                      _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                      ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_rejection_ex", rc)
    return Result(out_tokens, accept_len, dev_status, None, out_probs)


def spec_verify_tree_ex(logits: torch.Tensor, node_tokens: torch.Tensor, parents: torch.Tensor, *,
                        temperatures=None, temperature: float = 1.0, threshold_single: float = 1.0,
                        threshold_acc: float = 1.0, top_k=None, top_p=None, seed: int = 0,
                        offset: int = 0, out_tokens=None,
                        accept_index=None, accept_len=None, workspace=None, dev_status=None,
                        stream=None) -> Result:
    """spec_verify_tree where a request with temperature 0 walks by argmax and the others by the
    target-only rule at their temperature, with relaxed thresholds."""
    lib = load_library()
    _check_dev("logits", logits)
    B, N, V = logits.shape
    _check_dev("node_tokens", node_tokens, torch.int32)
    _check_dev("parents", parents, torch.int32)
    dev = logits.device
    stream = stream or torch.cuda.current_stream(dev)
    opt = _options(temperatures, temperature, threshold_single, threshold_acc, B, dev, top_k, top_p)
    out_tokens = out_tokens if out_tokens is not None else torch.empty((B, N), dtype=torch.int32, device=dev)
    accept_index = accept_index if accept_index is not None else torch.empty((B, N), dtype=torch.int32, device=dev)
    accept_len = accept_len if accept_len is not None else torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = spec_verify_workspace_bytes(MODE_TREE, B, N, V)
    workspace, dev_status = _ws_and_status(nbytes, dev, stream, workspace, dev_status)
    rc = lib.spec_verify_tree_ex(_ptr(logits), _logits_dtype(logits), _ptr(node_tokens),
                                 _ptr(parents), B, N, V, ctypes.byref(opt), int(seed) & (2**64 - 1),
                                 int(offset) & (2**64 - 1), _ptr(out_tokens), _ptr(accept_index),
                                 _ptr(accept_len), _ptr(workspace), workspace.numel(),
                                 _ptr(dev_status), ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_tree_ex", rc)
    return Result(out_tokens, accept_len, dev_status, accept_index)


def spec_verify_plan_budget(conf: torch.Tensor, cost: torch.Tensor, num_drafts=None, *,
                            admitted=None, budget=None, best_rate=None, stream=None):
    """Adaptive verification budget: conf [B, K] float32, cost [B*K + 1] float64, num_drafts [B]
    int32 or None (CUDA tensors).  Returns (admitted [B] int32, budget [1] int32, best_rate [1]
    float64), all on the device."""
    lib = load_library()
    _check_dev("conf", conf, torch.float32)
    _check_dev("cost", cost, torch.float64)
    B, K = conf.shape
    if cost.numel() != B * K + 1:
        raise ValueError("cost must hold B*K + 1 entries")
    if num_drafts is not None:
        _check_dev("num_drafts", num_drafts, torch.int32)
    dev = conf.device
    stream = stream or torch.cuda.current_stream(dev)
    admitted = admitted if admitted is not None else torch.empty(B, dtype=torch.int32, device=dev)
    budget = budget if budget is not None else torch.empty(1, dtype=torch.int32, device=dev)
    best_rate = best_rate if best_rate is not None else torch.empty(1, dtype=torch.float64, device=dev)
    nbytes = int(lib.spec_verify_plan_budget_workspace_bytes(B, K))
    if nbytes == 0:
        raise ValueError("the budget planner takes B * K <= 16384 slots and K <= 64")
    # Not the verifiers' workspace: the planner overwrites its buffer, whose counter region the
    # verifiers need to stay zero.
    key = (dev.index, stream.cuda_stream)
    ws = _plan_ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        _plan_ws_cache[key] = ws
    rc = lib.spec_verify_plan_budget(_ptr(conf), _ptr(num_drafts), B, K, _ptr(cost), _ptr(admitted),
                                     _ptr(budget), _ptr(best_rate), _ptr(ws), ws.numel(),
                                     ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError("spec_verify_plan_budget", rc)
    return admitted, budget, best_rate
