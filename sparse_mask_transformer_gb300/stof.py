"""Python binding of libstof.so (include/stof.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of the method: it takes torch tensors (used only as device
memory) and the current CUDA stream, passes raw pointers through ctypes,
and raises StofError on a non-OK status.  The library must have been built
(``python -m sparse_mask_transformer_gb300.build``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libstof.so")
SYNTH_LIB_PATH = os.path.join(_PKG, "libstof_synth.so")

STOF_OK = 0
STOF_ERR_INVALID_ARG = 1
STOF_ERR_SHAPE = 2
STOF_ERR_DTYPE = 3
STOF_ERR_ALIGNMENT = 4
STOF_ERR_WORKSPACE = 5
STOF_ERR_UNSUPPORTED = 6
STOF_ERR_DEVICE = 7
STOF_ERR_CUDA = 8
STOF_ERR_NOT_SYNCED = 9

STOF_F16 = 0
STOF_BF16 = 1

STOF_KERNEL_AUTO = -1
STOF_KERNEL_ROWWISE = 0
STOF_KERNEL_BLOCKWISE = 1

STOF_DEVERR_LOOKBACK_TIMEOUT = 0x1
STOF_DEVERR_PIPE_TIMEOUT = 0x2
STOF_DEVERR_BAD_FORMAT = 0x4

EXPORTED = ["stof_encode_workspace_bytes", "stof_encode_mask", "stof_format_sync",
            "stof_select_kernel", "stof_mha_fwd", "stof_status_string", "stof_version",
            "stof_last_cuda_error", "stof_tune_workspace_bytes", "stof_tune", "stof_tune_lookup",
            "stof_tune_clear", "stof_tune_density_bucket", "stof_encode_mask_bits", "stof_oproj_fwd",
            "stof_encode_rules", "stof_check_bounded_wait", "stof_mha_plan", "stof_mha_fwd_plan",
            "stof_select_kernel_heads", "stof_oproj_ln_fwd", "stof_oproj_ln_workspace_bytes", "stof_ex2_fma",
            "stof_mha_fwd_cross"]

STOF_MAX_RULES = 64
INT32_MIN, INT32_MAX = -(1 << 31), (1 << 31) - 1

STOF_TUNE_CANDIDATES = 13

STOF_PLAN_FORCED = 0
STOF_PLAN_ANALYTIC = 1
STOF_PLAN_TUNED = 2


class StofError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: status {status} ({stof_status_string(status)})"
        if status == STOF_ERR_CUDA:
            msg += f": {stof_last_cuda_error()}"
        super().__init__(msg)


class stof_format(ctypes.Structure):
    _fields_ = [
        ("n_masks", ctypes.c_int32), ("lq", ctypes.c_int32), ("lk", ctypes.c_int32),
        ("bm", ctypes.c_int32), ("bn", ctypes.c_int32), ("n_tr", ctypes.c_int32),
        ("n_tc", ctypes.c_int32), ("synced", ctypes.c_int32),
        ("full_row_ptr", ctypes.c_void_p), ("full_col_idx", ctypes.c_void_p),
        ("part_row_ptr", ctypes.c_void_p), ("part_col_idx", ctypes.c_void_p),
        ("bitmaps", ctypes.c_void_p), ("counts_dev", ctypes.c_void_p), ("scratch", ctypes.c_void_p),
        ("n_full", ctypes.c_int64), ("n_part", ctypes.c_int64), ("nnz", ctypes.c_int64),
        ("device_error", ctypes.c_int64),
    ]


class stof_mask_rule(ctypes.Structure):
    _fields_ = [
        ("band_lo", ctypes.c_int32), ("band_hi", ctypes.c_int32),
        ("global_rows", ctypes.c_void_p), ("global_cols", ctypes.c_void_p), ("blocks", ctypes.c_void_p),
        ("block", ctypes.c_int32),
    ]


class stof_tune_result(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int), ("bn", ctypes.c_int), ("ms", ctypes.c_float), ("density", ctypes.c_double),
        ("stages", ctypes.c_int), ("persistent", ctypes.c_int), ("rows_per_warp", ctypes.c_int),
        ("exp_split", ctypes.c_int), ("softmax_warpgroups", ctypes.c_int),
        ("cand_kernel", ctypes.c_int * STOF_TUNE_CANDIDATES), ("cand_bn", ctypes.c_int * STOF_TUNE_CANDIDATES),
        ("cand_stages", ctypes.c_int * STOF_TUNE_CANDIDATES),
        ("cand_persistent", ctypes.c_int * STOF_TUNE_CANDIDATES),
        ("cand_rows_per_warp", ctypes.c_int * STOF_TUNE_CANDIDATES),
        ("cand_exp_split", ctypes.c_int * STOF_TUNE_CANDIDATES),
        ("cand_softmax_warpgroups", ctypes.c_int * STOF_TUNE_CANDIDATES),
        ("cand_ms", ctypes.c_float * STOF_TUNE_CANDIDATES),
    ]


class stof_plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("stages", ctypes.c_int), ("persistent", ctypes.c_int),
                ("source", ctypes.c_int), ("rows_per_warp", ctypes.c_int), ("exp_split", ctypes.c_int),
                ("softmax_warpgroups", ctypes.c_int)]


_lib = None
_synth = None


def load_library(path: str = LIB_PATH):
    """Loads libstof.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with python -m sparse_mask_transformer_gb300.build")
        lib = ctypes.CDLL(path)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.stof_encode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        lib.stof_encode_workspace_bytes.restype = sz
        lib.stof_encode_mask.argtypes = [P, i32, i32, i32, i32, i32, P, sz, ctypes.POINTER(stof_format), P]
        lib.stof_encode_mask.restype = i32
        lib.stof_encode_mask_bits.argtypes = [P, i32, i32, i32, i32, i32, P, sz, ctypes.POINTER(stof_format), P]
        lib.stof_encode_mask_bits.restype = i32
        lib.stof_encode_rules.argtypes = [ctypes.POINTER(stof_mask_rule), i32, i32, i32, i32, i32, P, sz,
                                          ctypes.POINTER(stof_format), P]
        lib.stof_encode_rules.restype = i32
        lib.stof_check_bounded_wait.argtypes = [P, ctypes.c_double, P]
        lib.stof_check_bounded_wait.restype = i32
        lib.stof_ex2_fma.argtypes = [P, P, i64, P]
        lib.stof_ex2_fma.restype = i32
        lib.stof_format_sync.argtypes = [ctypes.POINTER(stof_format), P]
        lib.stof_format_sync.restype = i32
        lib.stof_select_kernel.argtypes = [ctypes.c_double, i32, i32]
        lib.stof_select_kernel.restype = i32
        lib.stof_select_kernel_heads.argtypes = [ctypes.c_double, i32, i32, i64, ctypes.c_double]
        lib.stof_select_kernel_heads.restype = i32
        lib.stof_mha_fwd.argtypes = [P, P, P, i32, i32, i32, i32, i32, ctypes.c_float,
                                     ctypes.POINTER(stof_format), i64, i64, i32, P, P]
        lib.stof_mha_fwd.restype = i32
        lib.stof_mha_fwd_cross.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, ctypes.c_float,
                                           ctypes.POINTER(stof_format), i64, i64, i32, P, P]
        lib.stof_mha_fwd_cross.restype = i32
        lib.stof_mha_plan.argtypes = [ctypes.POINTER(stof_format), i32, i32, i32, i32, i32, ctypes.POINTER(stof_plan)]
        lib.stof_mha_plan.restype = i32
        lib.stof_mha_fwd_plan.argtypes = [P, P, P, i32, i32, i32, i32, i32, ctypes.c_float,
                                          ctypes.POINTER(stof_format), i64, i64, ctypes.POINTER(stof_plan), P, P]
        lib.stof_mha_fwd_plan.restype = i32
        lib.stof_status_string.argtypes = [i32]
        lib.stof_status_string.restype = ctypes.c_char_p
        lib.stof_version.argtypes = []
        lib.stof_version.restype = i32
        lib.stof_last_cuda_error.argtypes = []
        lib.stof_last_cuda_error.restype = ctypes.c_char_p
        lib.stof_oproj_fwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P]
        lib.stof_oproj_fwd.restype = i32
        lib.stof_oproj_ln_fwd.argtypes = [P, P, P, P, P, P, ctypes.c_float, i32, i32, i32, i32, i32, i32, P, P, sz,
                                          P, P]
        lib.stof_oproj_ln_fwd.restype = i32
        lib.stof_oproj_ln_workspace_bytes.argtypes = [i32, i32, i32]
        lib.stof_oproj_ln_workspace_bytes.restype = sz
        lib.stof_tune_workspace_bytes.argtypes = [i32, i32]
        lib.stof_tune_workspace_bytes.restype = sz
        lib.stof_tune.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, i32, ctypes.c_float, i64, i64, P, sz, P,
                                  ctypes.POINTER(stof_tune_result), P]
        lib.stof_tune.restype = i32
        lib.stof_tune_lookup.argtypes = [i32, i32, ctypes.c_double, ctypes.POINTER(stof_tune_result)]
        lib.stof_tune_lookup.restype = i32
        lib.stof_tune_clear.argtypes = []
        lib.stof_tune_clear.restype = None
        lib.stof_tune_density_bucket.argtypes = [ctypes.c_double]
        lib.stof_tune_density_bucket.restype = i32
        _lib = lib
    return _lib


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str):
    if status != STOF_OK:
        raise StofError(status, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return STOF_F16
    if t.dtype == torch.bfloat16:
        return STOF_BF16
    raise StofError(STOF_ERR_DTYPE, f"tensor dtype {t.dtype}")


def stof_version() -> int:
    return load_library().stof_version()


def stof_last_cuda_error() -> str:
    return load_library().stof_last_cuda_error().decode()


def stof_status_string(status: int) -> str:
    return load_library().stof_status_string(int(status)).decode()


def stof_encode_workspace_bytes(n_masks: int, lq: int, lk: int, bm: int, bn: int) -> int:
    return int(load_library().stof_encode_workspace_bytes(n_masks, lq, lk, bm, bn))


def stof_encode_mask(mask: torch.Tensor, bm: int, bn: int, workspace: torch.Tensor,
                     fmt: stof_format | None = None, stream=None) -> stof_format:
    """mask: uint8/bool [n_masks, lq, lk] on the device, or in pinned host
    memory (the encoder then reads it over the host link); workspace:
    device uint8 tensor."""
    if mask.dim() != 3 or not mask.is_contiguous() or mask.element_size() != 1:
        raise StofError(STOF_ERR_SHAPE, "stof_encode_mask: mask must be contiguous 1-byte [n_masks, lq, lk]")
    if not mask.is_cuda and not mask.is_pinned():
        raise StofError(STOF_ERR_INVALID_ARG, "stof_encode_mask: a host mask must be in pinned memory")
    fmt = fmt if fmt is not None else stof_format()
    n_masks, lq, lk = mask.shape
    _check(load_library().stof_encode_mask(
        mask.data_ptr(), n_masks, lq, lk, bm, bn, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), ctypes.byref(fmt), _stream(stream)),
        "stof_encode_mask")
    return fmt


def stof_encode_mask_bits(mask_bits: torch.Tensor, lk: int, bm: int, bn: int, workspace: torch.Tensor,
                          fmt: stof_format | None = None, stream=None) -> stof_format:
    """mask_bits: device uint8 [n_masks, lq, lk / 8], bit c of byte jb = key 8 jb + c."""
    if (mask_bits.dim() != 3 or not mask_bits.is_contiguous() or mask_bits.element_size() != 1
            or lk % 8 or mask_bits.shape[2] != lk // 8):
        raise StofError(STOF_ERR_SHAPE, "stof_encode_mask_bits: mask must be contiguous uint8 [n_masks, lq, lk/8]")
    fmt = fmt if fmt is not None else stof_format()
    n_masks, lq, _ = mask_bits.shape
    _check(load_library().stof_encode_mask_bits(
        mask_bits.data_ptr(), n_masks, lq, lk, bm, bn, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), ctypes.byref(fmt), _stream(stream)),
        "stof_encode_mask_bits")
    return fmt


def bitset_words(flags, device="cuda") -> torch.Tensor:
    """Bool/0-1 array of n flags -> device int32 tensor of ceil(n / 32) words,
    flag b at bit b % 32 of word b / 32 (the layout of stof_mask_rule's bitsets)."""
    import numpy as np
    f = np.asarray(flags, dtype=bool).ravel()
    packed = np.packbits(f, bitorder="little")
    packed = np.concatenate([packed, np.zeros((-len(packed)) % 4, dtype=np.uint8)])
    return torch.from_numpy(np.frombuffer(packed.tobytes(), dtype="<i4").copy()).to(device)


class MaskRule:
    """One parametric mask for stof_encode_rules: a band lo <= i - j <= hi,
    global rows and columns and a block pattern, each a device bitset
    (bitset_words) or None."""

    def __init__(self, band_lo: int = 1, band_hi: int = 0, global_rows: torch.Tensor | None = None,
                 global_cols: torch.Tensor | None = None, blocks: torch.Tensor | None = None, block: int = 0):
        self.band_lo, self.band_hi = int(band_lo), int(band_hi)
        self.global_rows, self.global_cols, self.blocks, self.block = global_rows, global_cols, blocks, int(block)

    def as_c(self) -> stof_mask_rule:
        ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        return stof_mask_rule(self.band_lo, self.band_hi, ptr(self.global_rows), ptr(self.global_cols),
                              ptr(self.blocks), self.block)


def stof_encode_rules(rules: list, lq: int, lk: int, bm: int, bn: int, workspace: torch.Tensor,
                      fmt: stof_format | None = None, stream=None) -> stof_format:
    """rules: one MaskRule per mask (its bitsets stay alive until the encode is done)."""
    arr = (stof_mask_rule * max(1, len(rules)))(*[r.as_c() for r in rules])
    fmt = fmt if fmt is not None else stof_format()
    _check(load_library().stof_encode_rules(
        arr, len(rules), lq, lk, bm, bn, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        ctypes.byref(fmt), _stream(stream)), "stof_encode_rules")
    return fmt


def stof_check_bounded_wait(device_error: torch.Tensor, seconds: float, stream=None) -> None:
    """device_error: device int64 tensor of one element; the call ORs
    STOF_DEVERR_PIPE_TIMEOUT into it after `seconds` of a wait that never ends."""
    _check(load_library().stof_check_bounded_wait(device_error.data_ptr(), float(seconds), _stream(stream)),
           "stof_check_bounded_wait")


def stof_ex2_fma(x: torch.Tensor, y: torch.Tensor, stream=None) -> None:
    """y = the block-wise kernels' FMA-pipe exp2 of x (device fp32, same length)."""
    if x.dtype != torch.float32 or y.dtype != torch.float32 or x.numel() != y.numel():
        raise ValueError("x and y must be fp32 tensors of the same size")
    _check(load_library().stof_ex2_fma(x.data_ptr(), y.data_ptr(), x.numel(), _stream(stream)), "stof_ex2_fma")


def stof_format_sync(fmt: stof_format, stream=None) -> stof_format:
    _check(load_library().stof_format_sync(ctypes.byref(fmt), _stream(stream)), "stof_format_sync")
    return fmt


def stof_select_kernel(density: float, seq_len: int, head_dim: int) -> int:
    return int(load_library().stof_select_kernel(float(density), int(seq_len), int(head_dim)))


def stof_select_kernel_heads(density: float, seq_len: int, head_dim: int, heads: int,
                             tiles_per_row: float = -1.0) -> int:
    return int(load_library().stof_select_kernel_heads(float(density), int(seq_len), int(head_dim), int(heads),
                                                       float(tiles_per_row)))


def stof_mha_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, fmt: stof_format, scale: float,
                 mask_stride_b: int, mask_stride_h: int, which: int, o: torch.Tensor,
                 stream=None) -> torch.Tensor:
    """q, k, v, o: device [B, H, L, d] fp16/bf16, contiguous."""
    if q.dim() != 4:
        raise StofError(STOF_ERR_SHAPE, "stof_mha_fwd: q must be [B, H, L, d]")
    for t in (q, k, v, o):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise StofError(STOF_ERR_SHAPE, "stof_mha_fwd: q, k, v, o must match and be contiguous")
    B, H, L, d = q.shape
    _check(load_library().stof_mha_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _dtype_code(q), B, H, L, d, float(scale),
        ctypes.byref(fmt), int(mask_stride_b), int(mask_stride_h), int(which), o.data_ptr(),
        _stream(stream)), "stof_mha_fwd")
    return o


def stof_mha_fwd_cross(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, fmt: stof_format, scale: float,
                       mask_stride_b: int, mask_stride_h: int, which: int, o: torch.Tensor,
                       stream=None) -> torch.Tensor:
    """q, o: device [B, H, Lq, d]; k, v: device [B, H, Lk, d]; fp16/bf16, contiguous."""
    if q.dim() != 4 or k.dim() != 4:
        raise StofError(STOF_ERR_SHAPE, "stof_mha_fwd_cross: q, k must be [B, H, L, d]")
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    if (o.shape != q.shape or k.shape != (B, H, Lk, d) or v.shape != k.shape
            or any(t.dtype != q.dtype or not t.is_contiguous() for t in (k, v, o)) or not q.is_contiguous()):
        raise StofError(STOF_ERR_SHAPE, "stof_mha_fwd_cross: q, o [B, H, Lq, d] and k, v [B, H, Lk, d], contiguous")
    _check(load_library().stof_mha_fwd_cross(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _dtype_code(q), B, H, Lq, Lk, d, float(scale),
        ctypes.byref(fmt), int(mask_stride_b), int(mask_stride_h), int(which), o.data_ptr(),
        _stream(stream)), "stof_mha_fwd_cross")
    return o


class MaskedAttention:
    """The usual sequence of library calls for one attention with a dense
    mask, for PyTorch callers: stof_encode_mask into a workspace this object
    keeps (and grows when a larger one is needed), stof_format_sync, then
    stof_mha_fwd_cross.  No arithmetic here; every step is a library call.
    Reuse one object per stream: its workspace holds the last format."""

    def __init__(self, bm: int = 128, bn: int = 128):
        self.bm, self.bn = bm, bn
        self.workspace = None
        self.fmt = None

    def encode(self, mask: torch.Tensor, stream=None, device=None) -> stof_format:
        """mask: [n_masks, Lq, Lk], nonzero = valid, on the device or in
        pinned host memory (read by the encoder over the host link, with no
        device copy).  The workspace goes on the mask's device; for a host
        mask on `device` (default: the current CUDA device)."""
        n_masks, lq, lk = mask.shape
        need = stof_encode_workspace_bytes(n_masks, lq, lk, self.bm, self.bn)
        if need == 0:
            raise StofError(STOF_ERR_SHAPE, "MaskedAttention: bad mask or tile sizes")
        if mask.is_cuda:
            device = mask.device
        elif device is None:
            device = torch.device("cuda", torch.cuda.current_device())
        if self.workspace is None or self.workspace.numel() < need or self.workspace.device != device:
            self.workspace = torch.empty(need, dtype=torch.uint8, device=device)
        if mask.dtype in (torch.uint8, torch.bool) and mask.is_contiguous():
            m = mask
        elif mask.is_cuda:
            m = mask.to(torch.uint8).contiguous()
        else:
            raise StofError(STOF_ERR_SHAPE, "MaskedAttention: a host mask must be contiguous uint8 or bool")
        self.fmt = stof_encode_mask(m, self.bm, self.bn, self.workspace, stream=stream)
        return stof_format_sync(self.fmt, stream)

    def __call__(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor | None = None,
                 scale: float | None = None, mask_stride_b: int | None = None, mask_stride_h: int | None = None,
                 which: int = STOF_KERNEL_AUTO, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """q [B, H, Lq, d], k and v [B, H, Lk, d]; mask [n_masks, Lq, Lk]
        (None: the last encoded one).  Head (b, h) uses mask
        b * mask_stride_b + h * mask_stride_h; by default one mask per
        (b, h) if there are B * H, one per head if H, one for all if 1.
        scale defaults to 1 / sqrt(d)."""
        if mask is not None:
            self.encode(mask, stream, q.device)
        if self.fmt is None:
            raise StofError(STOF_ERR_INVALID_ARG, "MaskedAttention: no mask encoded")
        B, H, _, d = q.shape
        if mask_stride_b is None or mask_stride_h is None:
            n = self.fmt.n_masks
            if n == B * H:
                sb, sh = H, 1
            elif n == H:
                sb, sh = 0, 1
            elif n == 1:
                sb, sh = 0, 0
            else:
                raise StofError(STOF_ERR_SHAPE, "MaskedAttention: give the mask strides for this mask count")
            mask_stride_b = sb if mask_stride_b is None else mask_stride_b
            mask_stride_h = sh if mask_stride_h is None else mask_stride_h
        o = out if out is not None else torch.empty_like(q)
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        return stof_mha_fwd_cross(q, k, v, self.fmt, scale, mask_stride_b, mask_stride_h, which, o, stream)


def stof_mha_plan(fmt: stof_format, B: int, H: int, L: int, d: int, which: int) -> stof_plan:
    """What stof_mha_fwd would run for these sizes, format and kernel request."""
    plan = stof_plan()
    _check(load_library().stof_mha_plan(ctypes.byref(fmt), int(B), int(H), int(L), int(d), int(which),
                                        ctypes.byref(plan)), "stof_mha_plan")
    return plan


def stof_mha_fwd_plan(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, fmt: stof_format, scale: float,
                      mask_stride_b: int, mask_stride_h: int, plan: stof_plan, o: torch.Tensor,
                      stream=None) -> torch.Tensor:
    """stof_mha_fwd run exactly as `plan` says (kernel, ring depth, variant)."""
    if q.dim() != 4:
        raise StofError(STOF_ERR_SHAPE, "stof_mha_fwd_plan: q must be [B, H, L, d]")
    for t in (q, k, v, o):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise StofError(STOF_ERR_SHAPE, "stof_mha_fwd_plan: q, k, v, o must match and be contiguous")
    B, H, L, d = q.shape
    _check(load_library().stof_mha_fwd_plan(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _dtype_code(q), B, H, L, d, float(scale),
        ctypes.byref(fmt), int(mask_stride_b), int(mask_stride_h), ctypes.byref(plan), o.data_ptr(),
        _stream(stream)), "stof_mha_fwd_plan")
    return o


def stof_oproj_fwd(o: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None, residual: torch.Tensor | None,
                   y: torch.Tensor, device_error: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """o: device [B, H, L, d]; w: [N, H*d]; bias: [N] or None; residual: [B, L, N] or None;
    y: [B, L, N] (written).  device_error: optional device int64 tensor of one element."""
    if o.dim() != 4:
        raise StofError(STOF_ERR_SHAPE, "stof_oproj_fwd: o must be [B, H, L, d]")
    B, H, L, d = o.shape
    N = w.shape[0]
    if w.shape != (N, H * d) or y.shape != (B, L, N):
        raise StofError(STOF_ERR_SHAPE, "stof_oproj_fwd: w must be [N, H*d] and y [B, L, N]")
    for t in (o, w, y, bias, residual):
        if t is not None and (t.dtype != o.dtype or not t.is_contiguous()):
            raise StofError(STOF_ERR_SHAPE, "stof_oproj_fwd: tensors must share o's dtype and be contiguous")
    if bias is not None and bias.shape != (N,):
        raise StofError(STOF_ERR_SHAPE, "stof_oproj_fwd: bias must be [N]")
    if residual is not None and residual.shape != (B, L, N):
        raise StofError(STOF_ERR_SHAPE, "stof_oproj_fwd: residual must be [B, L, N]")
    ptr = lambda t: None if t is None else t.data_ptr()
    _check(load_library().stof_oproj_fwd(
        o.data_ptr(), w.data_ptr(), ptr(bias), ptr(residual), _dtype_code(o), B, H, L, d, N, y.data_ptr(),
        ptr(device_error), _stream(stream)), "stof_oproj_fwd")
    return y


def stof_oproj_ln_workspace_bytes(B: int, L: int, N: int) -> int:
    return int(load_library().stof_oproj_ln_workspace_bytes(int(B), int(L), int(N)))


def stof_oproj_ln_fwd(o: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None, residual: torch.Tensor | None,
                      gamma: torch.Tensor | None, beta: torch.Tensor | None, eps: float, y: torch.Tensor,
                      workspace: torch.Tensor, device_error: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """stof_oproj_fwd followed by a LayerNorm over the N features (gamma, beta: [N] or None);
    workspace: device tensor of at least stof_oproj_ln_workspace_bytes(B, L, N) bytes."""
    if o.dim() != 4:
        raise StofError(STOF_ERR_SHAPE, "stof_oproj_ln_fwd: o must be [B, H, L, d]")
    B, H, L, d = o.shape
    N = w.shape[0]
    if w.shape != (N, H * d) or y.shape != (B, L, N):
        raise StofError(STOF_ERR_SHAPE, "stof_oproj_ln_fwd: w must be [N, H*d] and y [B, L, N]")
    for t in (o, w, y, bias, residual, gamma, beta):
        if t is not None and (t.dtype != o.dtype or not t.is_contiguous()):
            raise StofError(STOF_ERR_SHAPE, "stof_oproj_ln_fwd: tensors must share o's dtype and be contiguous")
    for t in (bias, gamma, beta):
        if t is not None and t.shape != (N,):
            raise StofError(STOF_ERR_SHAPE, "stof_oproj_ln_fwd: bias, gamma and beta must be [N]")
    if residual is not None and residual.shape != (B, L, N):
        raise StofError(STOF_ERR_SHAPE, "stof_oproj_ln_fwd: residual must be [B, L, N]")
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    _check(load_library().stof_oproj_ln_fwd(
        o.data_ptr(), w.data_ptr(), ptr(bias), ptr(residual), ptr(gamma), ptr(beta), float(eps), _dtype_code(o),
        B, H, L, d, N, y.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        ptr(device_error), _stream(stream)), "stof_oproj_ln_fwd")
    return y


def stof_tune_workspace_bytes(n_masks: int, L: int) -> int:
    return int(load_library().stof_tune_workspace_bytes(n_masks, L))


def stof_tune(mask: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
              mask_stride_b: int, mask_stride_h: int, workspace: torch.Tensor, o: torch.Tensor,
              stream=None) -> stof_tune_result:
    """mask: device uint8 [n_masks, L, L]; q, k, v, o: device [B, H, L, d]."""
    if mask.dim() != 3 or not mask.is_contiguous() or mask.element_size() != 1:
        raise StofError(STOF_ERR_SHAPE, "stof_tune: mask must be contiguous 1-byte [n_masks, L, L]")
    for t in (q, k, v, o):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise StofError(STOF_ERR_SHAPE, "stof_tune: q, k, v, o must match and be contiguous")
    B, H, L, d = q.shape
    res = stof_tune_result()
    _check(load_library().stof_tune(
        mask.data_ptr(), mask.shape[0], q.data_ptr(), k.data_ptr(), v.data_ptr(), _dtype_code(q), B, H, L, d,
        float(scale), int(mask_stride_b), int(mask_stride_h), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), o.data_ptr(), ctypes.byref(res), _stream(stream)),
        "stof_tune")
    return res


def stof_tune_lookup(L: int, d: int, density: float):
    """The cached stof_tune_result for (L, d, density bucket), or None."""
    res = stof_tune_result()
    return res if load_library().stof_tune_lookup(int(L), int(d), float(density), ctypes.byref(res)) else None


def stof_tune_clear() -> None:
    load_library().stof_tune_clear()


def stof_tune_density_bucket(density: float) -> int:
    return int(load_library().stof_tune_density_bucket(float(density)))


def format_arrays(fmt: stof_format, workspace: torch.Tensor, n_full: int | None = None,
                  n_part: int | None = None) -> dict:
    """Device views of the format's arrays (slices of the workspace tensor);
    counts default to the synced host copies."""
    base = workspace.data_ptr()
    n_rows = fmt.n_masks * fmt.n_tr
    n_full = fmt.n_full if n_full is None else n_full
    n_part = fmt.n_part if n_part is None else n_part
    wpt = (fmt.bm // 8) * (fmt.bn // 8)

    def view(ptr, count, dtype, esize):
        off = ptr - base
        return workspace[off:off + count * esize].view(dtype)

    return dict(
        full_row_ptr=view(fmt.full_row_ptr, n_rows + 1, torch.int32, 4),
        part_row_ptr=view(fmt.part_row_ptr, n_rows + 1, torch.int32, 4),
        full_col_idx=view(fmt.full_col_idx, n_full, torch.int32, 4),
        part_col_idx=view(fmt.part_col_idx, n_part, torch.int32, 4),
        bitmaps=view(fmt.bitmaps, n_part * wpt, torch.int64, 8).view(n_part, fmt.bm // 8, fmt.bn // 8),
    )


def _synth_lib():
    global _synth
    if _synth is None:
        if not os.path.exists(SYNTH_LIB_PATH):
            raise RuntimeError(f"{SYNTH_LIB_PATH} is missing: build it first")
        lib = ctypes.CDLL(SYNTH_LIB_PATH)
        lib.stof_synth_causal_bernoulli_mask.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
        lib.stof_synth_causal_bernoulli_mask.restype = ctypes.c_int
        lib.stof_synth_causal_bernoulli_mask_bits.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
        lib.stof_synth_causal_bernoulli_mask_bits.restype = ctypes.c_int
        lib.stof_synth_pack_bits.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p]
        lib.stof_synth_pack_bits.restype = ctypes.c_int
        _synth = lib
    return _synth


def stof_synth_causal_bernoulli_mask_bits(out: torch.Tensor, n_masks: int, L: int, seed: int,
                                          threshold: int, stream=None) -> torch.Tensor:
    """Bit-packed form of stof_synth_causal_bernoulli_mask: out uint8 [n_masks, L, L/8]."""
    assert out.numel() == n_masks * L * L // 8 and out.element_size() == 1 and out.is_contiguous()
    rc = _synth_lib().stof_synth_causal_bernoulli_mask_bits(out.data_ptr(), n_masks, L, seed, threshold,
                                                            _stream(stream))
    if rc != 0:
        raise RuntimeError(f"stof_synth_causal_bernoulli_mask_bits failed: {rc}")
    return out


def stof_synth_pack_bits(dense: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Device uint8 [..., n] (n % 8 == 0) -> bit-packed uint8 [..., n / 8]."""
    assert dense.element_size() == 1 and dense.is_contiguous() and dense.shape[-1] % 8 == 0
    if out is None:
        out = torch.empty(*dense.shape[:-1], dense.shape[-1] // 8, dtype=torch.uint8, device=dense.device)
    rc = _synth_lib().stof_synth_pack_bits(dense.data_ptr(), out.data_ptr(), dense.numel(), _stream(stream))
    if rc != 0:
        raise RuntimeError(f"stof_synth_pack_bits failed: {rc}")
    return out


def stof_synth_causal_bernoulli_mask(out: torch.Tensor, n_masks: int, L: int, seed: int,
                                     threshold: int, stream=None) -> torch.Tensor:
    """Device generator of seeded causal-Bernoulli masks (libstof_synth.so)."""
    assert out.numel() == n_masks * L * L and out.element_size() == 1 and out.is_contiguous()
    rc = _synth_lib().stof_synth_causal_bernoulli_mask(out.data_ptr(), n_masks, L, seed, threshold,
                                                       _stream(stream))
    if rc != 0:
        raise RuntimeError(f"stof_synth_causal_bernoulli_mask failed: {rc}")
    return out
