"""ctypes binding of libspecdec.so (see include/specdec.h for the full contract).

Argument marshalling only: tensors become device pointers, strides and sizes; every step runs in
the library's CUDA kernels.  Importing this module raises ImportError when the library has not
been built -- there is no fallback.  Host-detected errors raise SpecdecError; device-detected
errors land in the caller's ``status`` tensor (zero it before the call, read it when convenient).
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspecdec.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                      "(or python -m speculative_decoding_specdec_gb300._build)")
lib = ctypes.CDLL(LIB_PATH)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_CAPACITY, ERR_INPUT_RANGE, ERR_TIMEOUT = range(7)
F32, BF16 = 0, 1
MAX_DRAFT = 31
GREEDY_SCRATCH_BYTES = 73728   # SPECDEC_GREEDY_SCRATCH_BYTES
REALIGN_PDL = 1                # SPECDEC_REALIGN_PDL

c_i32p = ctypes.POINTER(ctypes.c_int32)


class KvView(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p),
                ("stride_layer", ctypes.c_longlong), ("stride_kv", ctypes.c_longlong),
                ("stride_row", ctypes.c_longlong), ("stride_head", ctypes.c_longlong),
                ("dtype", ctypes.c_int), ("layers", ctypes.c_int), ("rows", ctypes.c_int),
                ("heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("cap_cols", ctypes.c_int)]


class RealignArgs(ctypes.Structure):
    _fields_ = [("src", KvView), ("dst", KvView), ("B", ctypes.c_int), ("D", ctypes.c_int),
                ("pad_id", ctypes.c_int32), ("copy_engine", ctypes.c_int),
                ("n_committed", ctypes.c_void_p), ("width", ctypes.c_void_p),
                ("accept_len", ctypes.c_void_p), ("out_token", ctypes.c_void_p),
                ("draft", ctypes.c_void_p), ("ids_src", ctypes.c_void_p),
                ("ids_dst", ctypes.c_void_p), ("mask_dst", ctypes.c_void_p),
                ("pos_dst", ctypes.c_void_p), ("n_committed_dst", ctypes.c_void_p),
                ("width_dst", ctypes.c_void_p), ("dev_status", ctypes.c_void_p),
                ("flags", ctypes.c_int), ("schedule", ctypes.c_void_p)]


class PoolArgs(ctypes.Structure):
    _fields_ = [("arena", KvView), ("scratch", KvView), ("n_rows", ctypes.c_int),
                ("D", ctypes.c_int), ("pad_id", ctypes.c_int32), ("in_place", ctypes.c_int),
                ("rows", ctypes.c_void_p), ("slot_col", ctypes.c_void_p),
                ("slot_cap", ctypes.c_void_p), ("slot_len", ctypes.c_void_p),
                ("pool_ids", ctypes.c_void_p), ("ids_cap", ctypes.c_int),
                ("batch_len", ctypes.c_void_p), ("width", ctypes.c_void_p),
                ("scratch_ids", ctypes.c_void_p), ("scratch_mask", ctypes.c_void_p),
                ("scratch_pos", ctypes.c_void_p), ("accept_len", ctypes.c_void_p),
                ("out_token", ctypes.c_void_p), ("draft", ctypes.c_void_p),
                ("by_slot", ctypes.c_int), ("dev_status", ctypes.c_void_p),
                ("slot_state", ctypes.c_void_p), ("slot_limit", ctypes.c_void_p),
                ("eos_id", ctypes.c_int32), ("schedule", ctypes.c_void_p)]


class ScheduleArgs(ctypes.Structure):
    _fields_ = [("S", ctypes.c_int), ("batch_size", ctypes.c_int), ("window", ctypes.c_int),
                ("slot_state", ctypes.c_void_p), ("slot_len", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("batch_offsets", ctypes.c_void_p),
                ("batch_uniform", ctypes.c_void_p), ("finished", ctypes.c_void_p),
                ("finished_reason", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("dev_status", ctypes.c_void_p)]


class AdmitArgs(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int), ("S", ctypes.c_int), ("D", ctypes.c_int),
                ("ids_cap", ctypes.c_int), ("arena_cols", ctypes.c_int64),
                ("slots", ctypes.c_void_p), ("cols", ctypes.c_void_p), ("caps", ctypes.c_void_p),
                ("limits", ctypes.c_void_p), ("prompt_ids", ctypes.c_void_p),
                ("prompt_off", ctypes.c_void_p), ("slot_state", ctypes.c_void_p),
                ("slot_col", ctypes.c_void_p), ("slot_cap", ctypes.c_void_p),
                ("slot_len", ctypes.c_void_p), ("slot_limit", ctypes.c_void_p),
                ("pool_ids", ctypes.c_void_p), ("dev_status", ctypes.c_void_p)]


SLOT_FREE, SLOT_ACTIVE, SLOT_FINISHED_EOS, SLOT_FINISHED_LENGTH = range(4)


_vp, _ll, _i, _f = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_float
lib.specdec_version.restype = _i
lib.specdec_version.argtypes = []
lib.specdec_status_string.restype = ctypes.c_char_p
lib.specdec_status_string.argtypes = [_i]
lib.specdec_wait_selftest.restype = _i
lib.specdec_wait_selftest.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _vp, _vp]
_sz = ctypes.c_size_t
lib.specdec_verify_greedy.restype = _i
lib.specdec_verify_greedy.argtypes = [_vp, _i, _i, _i, _i, _ll, _vp, _vp, _vp, _vp, _sz, _vp, _vp]
lib.specdec_verify_greedy_workspace.restype = _sz
lib.specdec_verify_greedy_workspace.argtypes = [_i, _i]
lib.specdec_verify_greedy_noalloc.restype = _i
lib.specdec_verify_greedy_noalloc.argtypes = [_vp, _i, _i, _i, _i, _ll, _vp, _vp, _vp, _vp, _vp]
lib.specdec_realign.restype = _i
lib.specdec_realign.argtypes = [ctypes.POINTER(RealignArgs), _vp]
lib.specdec_realign_inplace.restype = _i
lib.specdec_realign_inplace.argtypes = [ctypes.POINTER(RealignArgs), _vp]
lib.specdec_group_by_length.restype = _i
lib.specdec_group_by_length.argtypes = [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
lib.specdec_pool_gather.restype = _i
lib.specdec_pool_gather.argtypes = [ctypes.POINTER(PoolArgs), _vp]
lib.specdec_pool_append.restype = _i
lib.specdec_pool_append.argtypes = [ctypes.POINTER(PoolArgs), _vp]
if hasattr(lib, "specdec_verify_sample"):
    lib.specdec_verify_sample.restype = _i
    lib.specdec_verify_sample.argtypes = [_vp, _vp, _i, _i, _i, _i, _ll, _f, _vp, _vp, _vp, _vp,
                                          _vp, _vp, _vp, _vp]
lib.specdec_philox_uniforms.restype = _i
lib.specdec_philox_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint64, _i, _i, _vp, _vp]
lib.specdec_verify_sample_philox.restype = _i
lib.specdec_verify_sample_philox.argtypes = [_vp, _vp, _i, _i, _i, _i, _ll, _f, _vp,
                                             ctypes.c_uint64, ctypes.c_uint64, _vp, _vp, _vp,
                                             _vp, _vp, _vp]
lib.specdec_sampling_filter.restype = _i
lib.specdec_sampling_filter.argtypes = [_vp, _vp, _i, _i, _i, _i, _ll, _f, _i, _f, _vp, _vp, _vp]
lib.specdec_pool_schedule.restype = _i
lib.specdec_pool_schedule.argtypes = [ctypes.POINTER(ScheduleArgs), _vp]
lib.specdec_pool_admit.restype = _i
lib.specdec_pool_admit.argtypes = [ctypes.POINTER(AdmitArgs), _vp]
_i64, _i64p = ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)
lib.specdec_arena_create.restype = _i
lib.specdec_arena_create.argtypes = [_i64, ctypes.POINTER(_vp)]
lib.specdec_arena_destroy.restype = None
lib.specdec_arena_destroy.argtypes = [_vp]
lib.specdec_arena_alloc.restype = _i
lib.specdec_arena_alloc.argtypes = [_vp, _i64, _i64p]
lib.specdec_arena_free.restype = _i
lib.specdec_arena_free.argtypes = [_vp, _i64]
lib.specdec_arena_stats.restype = _i
lib.specdec_arena_stats.argtypes = [_vp, _i64p, _i64p, _i64p]


class KeepBound(ctypes.Structure):
    """specdec_keep_bound: the last kept token of a row under the sampling settings."""
    _fields_ = [("key", ctypes.c_uint32), ("index", ctypes.c_int32)]


class SpecdecError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {status_string(code)} (status {code})")
        self.code = code


def version() -> int:
    return lib.specdec_version()


def status_string(code: int) -> str:
    return lib.specdec_status_string(int(code)).decode()


def wait_selftest(polls, sleep_ns, status, stream=None):
    """Run the library's bounded wait on a barrier nothing completes (at most ``polls`` polls of
    about ``sleep_ns`` ns); it records ERR_TIMEOUT in ``status`` (int32 CUDA tensor)."""
    _need(status, torch.int32, "status")
    _check(lib.specdec_wait_selftest(int(polls), int(sleep_ns), _ptr(status), _stream(stream)),
           "specdec_wait_selftest")


def _check(rc, what):
    if rc != OK:
        raise SpecdecError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise ValueError(f"unsupported dtype {dt}")


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")


def kv_view(t: torch.Tensor) -> KvView:
    """View of a cache tensor shaped [L, 2, rows, H, cap, head_dim] whose last two dims are
    contiguous (a column of a head is contiguous and columns follow each other)."""
    if t.dim() != 6 or t.shape[1] != 2:
        raise ValueError("cache must be [L, 2, rows, H, cap, head_dim]")
    L, _, R, H, S, hd = t.shape
    if t.stride(5) != 1 or t.stride(4) != hd:
        raise ValueError("cache columns must be contiguous")
    return KvView(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2), t.stride(3),
                  dtype_code(t.dtype), L, R, H, hd, S)


def _score_rows(x, B, rows, name):
    """(row_stride) of a [B, rows, V] score tensor whose rows are evenly spaced."""
    if x.dim() != 3 or x.shape[0] != B or x.shape[1] != rows:
        raise ValueError(f"{name}: expected [B, {rows}, V], got {tuple(x.shape)}")
    if x.stride(2) != 1 or (B > 1 and x.stride(0) != rows * x.stride(1)):
        raise ValueError(f"{name}: rows must be evenly spaced with unit element stride")
    return x.stride(1)


def greedy_workspace_bytes(B, D) -> int:
    """Workspace bytes greedy verification needs for B rows of D drafts."""
    return int(lib.specdec_verify_greedy_workspace(int(B), int(D)))


def _workspace(ws, need, name):
    if ws is None or ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError(f"{name}: workspace must be a contiguous CUDA uint8 tensor")
    if ws.numel() < need:
        raise ValueError(f"{name}: workspace of {ws.numel()} bytes, {need} needed")
    return ctypes.c_void_p(ws.data_ptr()), ws.numel()


def verify_greedy(logits, draft, accept_len, out_token, status, workspace, stream=None):
    """Greedy verification: logits [B, D+1, V] (fp32/bf16), draft [B, D] int32 ->
    accept_len[B], out_token[B] int32 (written asynchronously on ``stream``).  ``workspace``: a
    zero-filled uint8 CUDA tensor of at least greedy_workspace_bytes(B, D) bytes; every call leaves
    it zero-filled again, so it is reused as is."""
    B, D = draft.shape
    V = logits.shape[-1]
    rs = _score_rows(logits, B, D + 1, "logits")
    for t, n in ((draft, "draft"), (accept_len, "accept_len"), (out_token, "out_token"),
                 (status, "status")):
        _need(t, torch.int32, n)
    wp, wn = _workspace(workspace, greedy_workspace_bytes(B, D) if B else 0,
                        "verify_greedy")
    _check(lib.specdec_verify_greedy(_ptr(logits), dtype_code(logits.dtype), B, D, V, rs,
                                     _ptr(draft), _ptr(accept_len), _ptr(out_token), wp, wn,
                                     _ptr(status), _stream(stream)), "specdec_verify_greedy")


def verify_greedy_noalloc(logits, draft, accept_len, out_token, status, stream=None):
    """Greedy verification on the library's static per-device scratch instead of a workspace
    (for callers that cannot allocate or keep a device buffer).  Calls that may overlap on one
    device share that scratch: keep them on one stream."""
    B, D = draft.shape
    V = logits.shape[-1]
    rs = _score_rows(logits, B, D + 1, "logits")
    for t, n in ((draft, "draft"), (accept_len, "accept_len"), (out_token, "out_token"),
                 (status, "status")):
        _need(t, torch.int32, n)
    _check(lib.specdec_verify_greedy_noalloc(_ptr(logits), dtype_code(logits.dtype), B, D, V, rs,
                                             _ptr(draft), _ptr(accept_len), _ptr(out_token),
                                             _ptr(status), _stream(stream)),
           "specdec_verify_greedy_noalloc")


def sampling_filter(target_logits, draft_logits, temperature, top_k, top_p, keep_bounds, status,
                    stream=None):
    """Top-k / top-p keep bounds of every score row into ``keep_bounds``, an int32 CUDA tensor
    [B, 2D+1, 2] holding specdec_keep_bound (key bits, index) per row."""
    B, Dp1 = target_logits.shape[0], target_logits.shape[1]
    D = Dp1 - 1
    V = target_logits.shape[-1]
    rs = _score_rows(target_logits, B, D + 1, "target_logits")
    rs2 = _score_rows(draft_logits, B, D, "draft_logits")
    if rs != rs2 or draft_logits.dtype != target_logits.dtype or draft_logits.shape[-1] != V:
        raise ValueError("target and draft scores must share dtype, V and row stride")
    _need(keep_bounds, torch.int32, "keep_bounds")
    _need(status, torch.int32, "status")
    if tuple(keep_bounds.shape) != (B, 2 * D + 1, 2) or not keep_bounds.is_contiguous():
        raise ValueError("keep_bounds must be a contiguous [B, 2D+1, 2] int32 tensor")
    _check(lib.specdec_sampling_filter(_ptr(target_logits), _ptr(draft_logits),
                                       dtype_code(target_logits.dtype), B, D, V, rs,
                                       float(temperature), int(top_k), float(top_p),
                                       _ptr(keep_bounds), _ptr(status), _stream(stream)),
           "specdec_sampling_filter")


def verify_sample(target_logits, draft_logits, draft, uniforms, temperature, accept_len,
                  out_token, status, residual=None, stream=None, keep_bounds=None):
    """Sampled verification (min(1, p/q) acceptance, normalised max(0, p - q) residual draw);
    ``keep_bounds`` from sampling_filter applies top-k / top-p."""
    B, D = draft.shape
    V = target_logits.shape[-1]
    rs = _score_rows(target_logits, B, D + 1, "target_logits")
    rs2 = _score_rows(draft_logits, B, D, "draft_logits")
    if rs != rs2 or draft_logits.dtype != target_logits.dtype or draft_logits.shape[-1] != V:
        raise ValueError("target and draft scores must share dtype, V and row stride")
    _need(uniforms, torch.float32, "uniforms")
    if tuple(uniforms.shape) != (B, D + 1) or not uniforms.is_contiguous():
        raise ValueError("uniforms must be a contiguous [B, D+1] float32 tensor")
    if residual is not None:
        _need(residual, torch.float32, "residual")
        if tuple(residual.shape) != (B, V) or not residual.is_contiguous():
            raise ValueError("residual must be a contiguous [B, V] float32 tensor")
    _check(lib.specdec_verify_sample(_ptr(target_logits), _ptr(draft_logits),
                                     dtype_code(target_logits.dtype), B, D, V, rs,
                                     float(temperature), _ptr(draft), _ptr(uniforms),
                                     _ptr(accept_len), _ptr(out_token), _ptr(residual),
                                     _ptr(keep_bounds), _ptr(status), _stream(stream)),
           "specdec_verify_sample")


def philox_uniforms(seed, offset, out, stream=None):
    """The uniforms [B, D+1] that verify_sample_philox draws for (seed, offset), into ``out``."""
    _need(out, torch.float32, "out")
    if out.dim() != 2 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, D+1] float32 tensor")
    B, Dp1 = out.shape
    _check(lib.specdec_philox_uniforms(int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1),
                                       B, Dp1 - 1, _ptr(out), _stream(stream)),
           "specdec_philox_uniforms")


def verify_sample_philox(target_logits, draft_logits, draft, seed, offset, temperature,
                         accept_len, out_token, status, residual=None, stream=None,
                         keep_bounds=None):
    """Sampled verification with the uniforms drawn in-kernel from (seed, offset) by
    Philox4x32-10 (see specdec.h); advance ``offset`` every round."""
    B, D = draft.shape
    V = target_logits.shape[-1]
    rs = _score_rows(target_logits, B, D + 1, "target_logits")
    rs2 = _score_rows(draft_logits, B, D, "draft_logits")
    if rs != rs2 or draft_logits.dtype != target_logits.dtype or draft_logits.shape[-1] != V:
        raise ValueError("target and draft scores must share dtype, V and row stride")
    if residual is not None:
        _need(residual, torch.float32, "residual")
        if tuple(residual.shape) != (B, V) or not residual.is_contiguous():
            raise ValueError("residual must be a contiguous [B, V] float32 tensor")
    _check(lib.specdec_verify_sample_philox(
        _ptr(target_logits), _ptr(draft_logits), dtype_code(target_logits.dtype), B, D, V, rs,
        float(temperature), _ptr(draft), int(seed) & (2 ** 64 - 1), int(offset) & (2 ** 64 - 1),
        _ptr(accept_len), _ptr(out_token), _ptr(residual), _ptr(keep_bounds), _ptr(status),
        _stream(stream)), "specdec_verify_sample_philox")


def _schedule(t):
    """Device address of a pair of scheduling words (None: fixed shares)."""
    if t is None:
        return None
    _need(t, torch.int32, "schedule")
    if t.numel() < 2 or not t.is_contiguous():
        raise ValueError("schedule needs 2 contiguous int32 elements")
    return t.data_ptr()


def realign(src, dst, n_committed, width, accept_len, out_token, draft, ids_src, ids_dst,
            mask_dst, pos_dst, n_committed_dst, width_dst, status, pad_id=0, copy_engine=0,
            pdl=False, stream=None, schedule=None):
    """EQSPEC realignment from cache ``src`` into cache ``dst`` (both [L, 2, B, H, cap, hd]).
    Passing the same tensor as ``src`` and ``dst`` moves the K/V in place
    (specdec_realign_inplace); the metadata outputs stay separate.  ``pdl`` launches it as a
    programmatic dependent of the kernel ahead of it (SPECDEC_REALIGN_PDL).  ``schedule``: None
    (fixed equal shares per CTA) or a zero-filled int32 CUDA tensor of 2 elements that the call
    leaves zero (work items taken from a counter; calls on other streams need their own)."""
    B, D = draft.shape
    in_place = src.data_ptr() == dst.data_ptr()
    a = RealignArgs()
    a.src = kv_view(src)
    a.dst = kv_view(dst)
    a.B, a.D, a.pad_id, a.copy_engine = B, D, int(pad_id), int(copy_engine)
    a.flags = REALIGN_PDL if pdl else 0
    a.schedule = _schedule(schedule)
    for name, t in (("n_committed", n_committed), ("width", width), ("accept_len", accept_len),
                    ("out_token", out_token), ("draft", draft), ("ids_src", ids_src),
                    ("ids_dst", ids_dst), ("pos_dst", pos_dst),
                    ("n_committed_dst", n_committed_dst), ("width_dst", width_dst),
                    ("dev_status", status)):
        _need(t, torch.int32, name)
        setattr(a, name, t.data_ptr())
    _need(mask_dst, torch.uint8, "mask_dst")
    a.mask_dst = mask_dst.data_ptr()
    if ids_src.shape != (B, src.shape[4]) or not ids_src.is_contiguous():
        raise ValueError("ids_src must be a contiguous [B, src cap] int32 tensor")
    for t, n in ((ids_dst, "ids_dst"), (mask_dst, "mask_dst"), (pos_dst, "pos_dst")):
        if t.shape != (B, dst.shape[4]) or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous [B, dst cap] tensor")
    if in_place:
        _check(lib.specdec_realign_inplace(ctypes.byref(a), _stream(stream)),
               "specdec_realign_inplace")
    else:
        _check(lib.specdec_realign(ctypes.byref(a), _stream(stream)), "specdec_realign")


def group_by_length(lengths, batch_size, max_len, perm, batch_offsets, batch_uniform,
                    num_batches, num_uniform, status, stream=None):
    """EXSPEC grouping of pool rows by length (stable counting sort, uniform batches first)."""
    N = lengths.numel()
    for t, n in ((lengths, "lengths"), (perm, "perm"), (batch_offsets, "batch_offsets"),
                 (num_batches, "num_batches"), (num_uniform, "num_uniform"), (status, "status")):
        _need(t, torch.int32, n)
    _need(batch_uniform, torch.uint8, "batch_uniform")
    if perm.numel() < N or batch_offsets.numel() < N + 1 or batch_uniform.numel() < N:
        raise ValueError("output buffers too small")
    _check(lib.specdec_group_by_length(_ptr(lengths), N, int(batch_size), int(max_len),
                                       _ptr(perm), _ptr(batch_offsets), _ptr(batch_uniform),
                                       _ptr(num_batches), _ptr(num_uniform), _ptr(status),
                                       _stream(stream)), "specdec_group_by_length")


def _pool_args(arena, scratch, rows, D, slot_col, slot_cap, slot_len, pool_ids, batch_len, width,
               status, pad_id, in_place):
    a = PoolArgs()
    a.arena = kv_view(arena)
    a.scratch = kv_view(scratch)
    a.n_rows, a.D, a.pad_id, a.in_place = rows.numel(), int(D), int(pad_id), int(bool(in_place))
    for name, t in (("rows", rows), ("slot_col", slot_col), ("slot_cap", slot_cap),
                    ("slot_len", slot_len), ("pool_ids", pool_ids), ("batch_len", batch_len),
                    ("width", width), ("dev_status", status)):
        _need(t, torch.int32, name)
        setattr(a, name, t.data_ptr())
    if pool_ids.dim() != 2 or not pool_ids.is_contiguous():
        raise ValueError("pool_ids must be a contiguous [slots, ids_cap] int32 tensor")
    a.ids_cap = pool_ids.shape[1]
    return a


def pool_gather(arena, scratch, rows, D, slot_col, slot_cap, slot_len, pool_ids, batch_len, width,
                status, scratch_ids=None, scratch_mask=None, scratch_pos=None, pad_id=0,
                in_place=False, stream=None, schedule=None):
    """Gather pool slots ``rows`` into the padded batch buffer ``scratch`` (see specdec.h).
    ``schedule``: as in ``realign``."""
    a = _pool_args(arena, scratch, rows, D, slot_col, slot_cap, slot_len, pool_ids, batch_len,
                   width, status, pad_id, in_place)
    a.schedule = _schedule(schedule)
    if not in_place:
        for t, n, dt in ((scratch_ids, "scratch_ids", torch.int32),
                         (scratch_mask, "scratch_mask", torch.uint8),
                         (scratch_pos, "scratch_pos", torch.int32)):
            _need(t, dt, n)
            if t.shape != (scratch.shape[2], scratch.shape[4]) or not t.is_contiguous():
                raise ValueError(f"{n} must be a contiguous [rows, scratch cap] tensor")
        a.scratch_ids, a.scratch_mask, a.scratch_pos = (scratch_ids.data_ptr(),
                                                        scratch_mask.data_ptr(),
                                                        scratch_pos.data_ptr())
    _check(lib.specdec_pool_gather(ctypes.byref(a), _stream(stream)), "specdec_pool_gather")


def pool_append(arena, scratch, rows, D, slot_col, slot_cap, slot_len, pool_ids, batch_len, width,
                accept_len, out_token, draft, status, in_place=False, by_slot=False,
                slot_state=None, slot_limit=None, eos_id=-1, stream=None, schedule=None):
    """Append a verified batch back to its pool slots (see specdec.h).  With ``by_slot`` the
    accept lengths, tokens and drafts are pool-wide arrays indexed by slot.  With ``slot_state``
    (and ``slot_limit``) finished sequences are retired: end-of-sequence token ``eos_id`` or the
    length limit.  ``schedule``: as in ``realign``."""
    a = _pool_args(arena, scratch, rows, D, slot_col, slot_cap, slot_len, pool_ids, batch_len,
                   width, status, 0, in_place)
    a.schedule = _schedule(schedule)
    a.by_slot = int(bool(by_slot))
    for name, t in (("accept_len", accept_len), ("out_token", out_token), ("draft", draft)):
        _need(t, torch.int32, name)
        setattr(a, name, t.data_ptr())
    if slot_state is not None:
        _need(slot_state, torch.uint8, "slot_state")
        _need(slot_limit, torch.int32, "slot_limit")
        a.slot_state, a.slot_limit, a.eos_id = (slot_state.data_ptr(), slot_limit.data_ptr(),
                                                int(eos_id))
    _check(lib.specdec_pool_append(ctypes.byref(a), _stream(stream)), "specdec_pool_append")


# ------------------------------------------------------------------------ SequencePool lifecycle

def pool_schedule(slot_state, slot_len, batch_size, window, perm, batch_offsets, batch_uniform,
                  finished, finished_reason, counts, status, stream=None):
    """Group the ACTIVE slots by length window, list (and free) the finished ones; counts =
    {num_batches, num_windowed, num_active, num_finished} (see specdec.h)."""
    S = slot_state.numel()
    _need(slot_state, torch.uint8, "slot_state")
    _need(batch_uniform, torch.uint8, "batch_uniform")
    _need(finished_reason, torch.uint8, "finished_reason")
    for t, n in ((slot_len, "slot_len"), (perm, "perm"), (batch_offsets, "batch_offsets"),
                 (finished, "finished"), (counts, "counts"), (status, "status")):
        _need(t, torch.int32, n)
    if (slot_len.numel() < S or perm.numel() < S or batch_offsets.numel() < S + 1 or
            batch_uniform.numel() < S or finished.numel() < S or finished_reason.numel() < S or
            counts.numel() < 4):
        raise ValueError("buffers too small")
    a = ScheduleArgs()
    a.S, a.batch_size, a.window = S, int(batch_size), int(window)
    for name, t in (("slot_state", slot_state), ("slot_len", slot_len), ("perm", perm),
                    ("batch_offsets", batch_offsets), ("batch_uniform", batch_uniform),
                    ("finished", finished), ("finished_reason", finished_reason),
                    ("counts", counts), ("dev_status", status)):
        setattr(a, name, t.data_ptr())
    _check(lib.specdec_pool_schedule(ctypes.byref(a), _stream(stream)), "specdec_pool_schedule")


def pool_admit(slots, cols, caps, limits, prompt_ids, prompt_off, D, arena_cols, slot_state,
               slot_col, slot_cap, slot_len, slot_limit, pool_ids, status, stream=None):
    """Admit prompts (concatenated in ``prompt_ids``, bounds in ``prompt_off``) into FREE slots
    (see specdec.h)."""
    n = slots.numel()
    _need(slot_state, torch.uint8, "slot_state")
    for t, nm in ((slots, "slots"), (cols, "cols"), (caps, "caps"), (limits, "limits"),
                  (prompt_ids, "prompt_ids"), (prompt_off, "prompt_off"), (slot_col, "slot_col"),
                  (slot_cap, "slot_cap"), (slot_len, "slot_len"), (slot_limit, "slot_limit"),
                  (pool_ids, "pool_ids"), (status, "status")):
        _need(t, torch.int32, nm)
    if cols.numel() < n or caps.numel() < n or limits.numel() < n or prompt_off.numel() < n + 1:
        raise ValueError("per-entry arrays too small")
    if pool_ids.dim() != 2 or not pool_ids.is_contiguous():
        raise ValueError("pool_ids must be a contiguous [slots, ids_cap] int32 tensor")
    a = AdmitArgs()
    a.n, a.S, a.D, a.ids_cap = n, slot_state.numel(), int(D), pool_ids.shape[1]
    a.arena_cols = int(arena_cols)
    for name, t in (("slots", slots), ("cols", cols), ("caps", caps), ("limits", limits),
                    ("prompt_ids", prompt_ids), ("prompt_off", prompt_off),
                    ("slot_state", slot_state), ("slot_col", slot_col), ("slot_cap", slot_cap),
                    ("slot_len", slot_len), ("slot_limit", slot_limit), ("pool_ids", pool_ids),
                    ("dev_status", status)):
        setattr(a, name, t.data_ptr())
    _check(lib.specdec_pool_admit(ctypes.byref(a), _stream(stream)), "specdec_pool_admit")


class Arena:
    """Host first-fit allocator of arena columns (specdec_arena_*; no GPU involved)."""

    def __init__(self, cols: int):
        h = ctypes.c_void_p()
        _check(lib.specdec_arena_create(int(cols), ctypes.byref(h)), "specdec_arena_create")
        self._h = h
        self.cols = int(cols)

    def alloc(self, ncols: int):
        """Lowest free run of ``ncols`` columns, or None when none is free."""
        c = ctypes.c_int64()
        rc = lib.specdec_arena_alloc(self._h, int(ncols), ctypes.byref(c))
        if rc == ERR_CAPACITY:
            return None
        _check(rc, "specdec_arena_alloc")
        return c.value

    def free(self, col: int) -> None:
        _check(lib.specdec_arena_free(self._h, int(col)), "specdec_arena_free")

    def stats(self):
        """(free columns, largest free run, allocations)."""
        v = [ctypes.c_int64() for _ in range(3)]
        _check(lib.specdec_arena_stats(self._h, *[ctypes.byref(x) for x in v]),
               "specdec_arena_stats")
        return tuple(x.value for x in v)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib.specdec_arena_destroy(h)
            self._h = None
