"""Python binding of libpvl: argument marshalling only.

Every function checks shapes/dtypes, allocates outputs with torch on the
tensors' CUDA device when the caller passes none, and calls the C entry point
of the same name on the current torch stream.  All arithmetic runs in the
library's CUDA kernels; nothing here computes attention, seq_ids or tile maps.
"""

from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import numpy as np
import torch

from . import _lib

PVL_OK, PVL_ERR_INVALID_ARG, PVL_ERR_UNSUPPORTED, PVL_ERR_CUDA, PVL_ERR_TIMEOUT = range(5)
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT"}

TM_LEVELS = 2
TM_FIELDS = ["header", "q_nv", "q_lo", "q_hi", "k_nv", "k_lo", "k_hi", "cls", "row_count", "row_full",
             "row_list", "col_count", "col_full", "col_list", "q_order", "k_order"]
EMPTY, PARTIAL, FULL = 0, 1, 2


class PvlError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pvl {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _check(status: int) -> None:
    if status != PVL_OK:
        raise PvlError(status, _lib.load().pvl_last_error_message().decode())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need_cuda(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# ------------------------------------------------------------------ seq_ids
def pack_build_seq_ids(seg_frames, seg_valid, tokens_per_frame: int, L: int, out: torch.Tensor | None = None,
                       device=None, stream=None) -> torch.Tensor:
    """int32 [B, L] seq_id on the GPU from host [B, K] frame / valid-frame tables."""
    frames = np.ascontiguousarray(np.asarray(seg_frames, dtype=np.int32))
    valid = np.ascontiguousarray(np.asarray(seg_valid, dtype=np.int32))
    if frames.ndim != 2 or frames.shape != valid.shape:
        raise ValueError("seg_frames and seg_valid must both be [B, K]")
    B, K = frames.shape
    if out is None:
        out = torch.empty((B, L), dtype=torch.int32, device=device or "cuda")
    _need_cuda(out, "out", torch.int32, (B, L))
    with torch.cuda.device(out.device):
        _check(_lib.load().pack_build_seq_ids(frames.ctypes.data, valid.ctypes.data, B, K, int(tokens_per_frame),
                                              int(L), out.data_ptr(), _stream(stream)))
    return out


# ----------------------------------------------------------------- tile map
@dataclass
class TileMap:
    """Device workspace written by tile_map_build plus typed views of its arrays.

    Level 0 is the map at (block_m, block_n); level 1 the map at
    (2 * block_m, block_n) over pairs of query tiles.  L is the query length,
    Lk the key length (equal for self attention)."""
    ws: torch.Tensor
    B: int
    L: int
    block_m: int
    block_n: int
    offsets: tuple  # LEVELS * len(TM_FIELDS) byte offsets
    Lk: int = 0     # 0: same as L

    def __post_init__(self):
        if not self.Lk:
            self.Lk = self.L

    def blocks(self, level: int = 0):
        return (self.block_m * (2 if level else 1), self.block_n)

    def n_tiles(self, level: int = 0):
        bm, bn = self.blocks(level)
        return -(-self.L // bm), -(-self.Lk // bn)

    @property
    def nTq(self) -> int:
        return self.n_tiles(0)[0]

    @property
    def nTk(self) -> int:
        return self.n_tiles(0)[1]

    def field(self, name: str, level: int = 0) -> torch.Tensor:
        i = TM_FIELDS.index(name)
        B = self.B
        nq, nk = self.n_tiles(level)
        shapes = {"header": (16,), "q_nv": (B, nq), "q_lo": (B, nq), "q_hi": (B, nq), "k_nv": (B, nk),
                  "k_lo": (B, nk), "k_hi": (B, nk), "cls": (B, nq, nk), "row_count": (B, nq),
                  "row_full": (B, nq), "row_list": (B, nq, nk), "col_count": (B, nk), "col_full": (B, nk),
                  "col_list": (B, nk, nq), "q_order": (B * nq,), "k_order": (B * nk,)}
        shape = shapes[name]
        n = int(np.prod(shape))
        off = self.offsets[level * len(TM_FIELDS) + i]
        if name == "cls":
            return self.ws[off:off + n].view(shape)
        return self.ws[off:off + 4 * n].view(torch.int32).view(shape)

    def to_host(self, level: int = 0) -> dict:
        out = {name: self.field(name, level).cpu().numpy() for name in TM_FIELDS}
        bm, bn = self.blocks(level)
        nq, nk = self.n_tiles(level)
        out.update(B=self.B, L=self.L, Lk=self.Lk, block_m=bm, block_n=bn, nTq=nq, nTk=nk)
        return out


def tile_map_ws_bytes(B: int, L: int, block_m: int = 128, block_n: int = 128, Lk: int | None = None) -> int:
    if Lk is None:
        return int(_lib.load().tile_map_ws_bytes(B, L, block_m, block_n))
    return int(_lib.load().tile_map_ws_bytes_cross(B, L, Lk, block_m, block_n))


def tile_map_build(seq_id: torch.Tensor, block_m: int = 128, block_n: int = 128,
                   ws: torch.Tensor | None = None, stream=None, k_seq_id: torch.Tensor | None = None) -> TileMap:
    """Tile map of the seq_id mask; with k_seq_id (int32 [B, Lk]) the
    cross-attention map of queries with ids seq_id against keys with ids
    k_seq_id."""
    lib = _lib.load()
    if seq_id.dim() != 2:
        raise ValueError("seq_id must be [B, L]")
    _need_cuda(seq_id, "seq_id", torch.int32)
    B, L = seq_id.shape
    Lk = L
    if k_seq_id is not None:
        if k_seq_id.dim() != 2 or k_seq_id.shape[0] != B:
            raise ValueError("k_seq_id must be [B, Lk]")
        _need_cuda(k_seq_id, "k_seq_id", torch.int32)
        Lk = k_seq_id.shape[1]
    nbytes = int(lib.tile_map_ws_bytes_cross(B, L, Lk, block_m, block_n))
    if nbytes == 0:
        raise PvlError(PVL_ERR_INVALID_ARG, "bad tile map sizes")
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=seq_id.device)
    offs = (ctypes.c_size_t * (TM_LEVELS * len(TM_FIELDS)))()
    with torch.cuda.device(seq_id.device):
        if k_seq_id is None:
            _check(lib.tile_map_layout(B, L, block_m, block_n, ctypes.addressof(offs)))
            _check(lib.tile_map_build(seq_id.data_ptr(), B, L, block_m, block_n, ws.data_ptr(), ws.numel(),
                                      _stream(stream)))
        else:
            _check(lib.tile_map_layout_cross(B, L, Lk, block_m, block_n, ctypes.addressof(offs)))
            _check(lib.tile_map_build_cross(seq_id.data_ptr(), k_seq_id.data_ptr(), B, L, Lk, block_m, block_n,
                                            ws.data_ptr(), ws.numel(), _stream(stream)))
    return TileMap(ws, B, L, block_m, block_n, tuple(offs), Lk)


# ---------------------------------------------------------------- attention
def _qkv_shape(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("q must be [B, L, H, D]")
    return tuple(q.shape)


def _key_side(q, k, seq_id, k_seq_id, tile_map):
    """Checks the key-side shapes; returns (Lk, key ids)."""
    B, L, H, D = _qkv_shape(q)
    Lk = L if k_seq_id is None else int(k.shape[1]) if k.dim() == 4 else -1
    _need_cuda(seq_id, "seq_id", torch.int32, (B, L))
    if k_seq_id is not None:
        _need_cuda(k_seq_id, "k_seq_id", torch.int32, (B, Lk))
    if (tile_map.B, tile_map.L, tile_map.Lk) != (B, L, Lk):
        raise ValueError("tile map was built for another [B, Lq, Lk]")
    return Lk, (seq_id if k_seq_id is None else k_seq_id)


def masked_attn_fwd(q, k, v, seq_id, tile_map: TileMap, scale: float | None = None, o=None, lse=None,
                    stream=None, k_seq_id=None):
    """(O bf16 [B, L, H, D], LSE fp32 [B, H, L]) of seq_id-masked softmax attention.

    With k_seq_id (int32 [B, Lk]) it is cross attention: k and v are
    [B, Lk, H, D] and query i attends key j iff seq_id[i] == k_seq_id[j] >= 0."""
    B, L, H, D = _qkv_shape(q)
    Lk, kid = _key_side(q, k, seq_id, k_seq_id, tile_map)
    _need_cuda(q, "q", torch.bfloat16, (B, L, H, D))
    for name, t in (("k", k), ("v", v)):
        _need_cuda(t, name, torch.bfloat16, (B, Lk, H, D))
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    _need_cuda(o, "o", torch.bfloat16, (B, L, H, D))
    _need_cuda(lse, "lse", torch.float32, (B, H, L))
    lib = _lib.load()
    with torch.cuda.device(q.device):
        if k_seq_id is None:
            _check(lib.masked_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), seq_id.data_ptr(),
                                       tile_map.ws.data_ptr(), B, L, H, D, scale, o.data_ptr(), lse.data_ptr(),
                                       _stream(stream)))
        else:
            _check(lib.masked_attn_fwd_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), seq_id.data_ptr(),
                                             kid.data_ptr(), tile_map.ws.data_ptr(), B, L, Lk, H, D, scale,
                                             o.data_ptr(), lse.data_ptr(), _stream(stream)))
    return o, lse


def masked_attn_bwd_ws_bytes(B: int, L: int, H: int, D: int, Lk: int | None = None) -> int:
    if Lk is None:
        return int(_lib.load().masked_attn_bwd_ws_bytes(B, L, H, D))
    return int(_lib.load().masked_attn_bwd_ws_bytes_cross(B, L, Lk, H, D))


def masked_attn_bwd(q, k, v, o, do, lse, seq_id, tile_map: TileMap, scale: float | None = None, dq=None,
                    dk=None, dv=None, ws=None, stream=None, k_seq_id=None):
    """(dQ, dK, dV) of the masked attention, from the saved LSE: dQ like q,
    dK and dV like k (cross attention with k_seq_id, as masked_attn_fwd)."""
    B, L, H, D = _qkv_shape(q)
    Lk, kid = _key_side(q, k, seq_id, k_seq_id, tile_map)
    for name, t in (("q", q), ("o", o), ("do", do)):
        _need_cuda(t, name, torch.bfloat16, (B, L, H, D))
    for name, t in (("k", k), ("v", v)):
        _need_cuda(t, name, torch.bfloat16, (B, Lk, H, D))
    _need_cuda(lse, "lse", torch.float32, (B, H, L))
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    _need_cuda(dq, "dq", torch.bfloat16, (B, L, H, D))
    for name, t in (("dk", dk), ("dv", dv)):
        _need_cuda(t, name, torch.bfloat16, (B, Lk, H, D))
    lib = _lib.load()
    nbytes = int(lib.masked_attn_bwd_ws_bytes_cross(B, L, Lk, H, D))
    if ws is None:
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        if k_seq_id is None:
            _check(lib.masked_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                       lse.data_ptr(), seq_id.data_ptr(), tile_map.ws.data_ptr(), B, L, H, D,
                                       scale, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                                       ws.numel(), _stream(stream)))
        else:
            _check(lib.masked_attn_bwd_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                             lse.data_ptr(), seq_id.data_ptr(), kid.data_ptr(),
                                             tile_map.ws.data_ptr(), B, L, Lk, H, D, scale, dq.data_ptr(),
                                             dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), ws.numel(),
                                             _stream(stream)))
    return dq, dk, dv


def masked_attn_bwd_no_alloc(q, k, v, o, do, lse, seq_id, tile_map: TileMap, scale: float | None = None,
                             dq=None, dk=None, dv=None, stream=None):
    """masked_attn_bwd without a workspace argument, for callers that must not
    allocate device memory: the scratch is the library's own static device
    array (limit PVL_NO_ALLOC_SCRATCH_BYTES).  Pass dq/dk/dv to avoid the
    output allocations too.  Calls that overlap on the GPU share that scratch
    and must be serialised."""
    B, L, H, D = _qkv_shape(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _need_cuda(t, name, torch.bfloat16, (B, L, H, D))
    _need_cuda(lse, "lse", torch.float32, (B, H, L))
    _need_cuda(seq_id, "seq_id", torch.int32, (B, L))
    if (tile_map.B, tile_map.L) != (B, L):
        raise ValueError("tile map was built for another [B, L]")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _need_cuda(t, name, torch.bfloat16, (B, L, H, D))
    with torch.cuda.device(q.device):
        _check(_lib.load().masked_attn_bwd_no_alloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            seq_id.data_ptr(), tile_map.ws.data_ptr(), B, L, H, D, scale, dq.data_ptr(), dk.data_ptr(),
            dv.data_ptr(), _stream(stream)))
    return dq, dk, dv


# -------------------------------------------------------------------- AdaLN
def adaln_fwd(x, shift, scale, eps: float = 1e-6, y=None, stats: bool = False, stream=None):
    """y = layer_norm(x) * (1 + scale) + shift ("AdaptiveLoad" §2.B): x bf16
    [B, N, D], shift / scale fp32 [B, D].  Returns y, or (y, mean, rstd) with
    stats=True."""
    if x.dim() != 3:
        raise ValueError("x must be [B, N, D]")
    B, N, D = x.shape
    _need_cuda(x, "x", torch.bfloat16, (B, N, D))
    _need_cuda(shift, "shift", torch.float32, (B, D))
    _need_cuda(scale, "scale", torch.float32, (B, D))
    y = torch.empty_like(x) if y is None else y
    _need_cuda(y, "y", torch.bfloat16, (B, N, D))
    mean = rstd = None
    if stats:
        mean = torch.empty((B, N), dtype=torch.float32, device=x.device)
        rstd = torch.empty((B, N), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        _check(_lib.load().adaln_fwd(x.data_ptr(), shift.data_ptr(), scale.data_ptr(), B, N, D, float(eps),
                                     y.data_ptr(), _ptr(mean), _ptr(rstd), _stream(stream)))
    return (y, mean, rstd) if stats else y


def adaln_bwd_ws_bytes(B: int, N: int, D: int) -> int:
    return int(_lib.load().adaln_bwd_ws_bytes(B, N, D))


def adaln_bwd(x, scale, dy, eps: float = 1e-6, dx=None, dshift=None, dscale=None, ws=None, stream=None):
    """(dx bf16 [B, N, D], dshift fp32 [B, D], dscale fp32 [B, D]) of adaln_fwd."""
    if x.dim() != 3:
        raise ValueError("x must be [B, N, D]")
    B, N, D = x.shape
    _need_cuda(x, "x", torch.bfloat16, (B, N, D))
    _need_cuda(dy, "dy", torch.bfloat16, (B, N, D))
    _need_cuda(scale, "scale", torch.float32, (B, D))
    dx = torch.empty_like(x) if dx is None else dx
    dshift = torch.empty((B, D), dtype=torch.float32, device=x.device) if dshift is None else dshift
    dscale = torch.empty((B, D), dtype=torch.float32, device=x.device) if dscale is None else dscale
    _need_cuda(dx, "dx", torch.bfloat16, (B, N, D))
    _need_cuda(dshift, "dshift", torch.float32, (B, D))
    _need_cuda(dscale, "dscale", torch.float32, (B, D))
    lib = _lib.load()
    nbytes = int(lib.adaln_bwd_ws_bytes(B, N, D))
    if ws is None:
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        _check(lib.adaln_bwd(x.data_ptr(), scale.data_ptr(), dy.data_ptr(), B, N, D, float(eps), dx.data_ptr(),
                             dshift.data_ptr(), dscale.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return dx, dshift, dscale


# ------------------------------------------------------------ masked loss
def masked_mse_ws_bytes(B: int, L: int, C: int) -> int:
    return int(_lib.load().masked_mse_ws_bytes(B, L, C))


def _loss_args(pred, target, seq_id):
    if pred.dim() != 3:
        raise ValueError("pred must be [B, L, C]")
    B, L, C = pred.shape
    _need_cuda(pred, "pred", torch.bfloat16, (B, L, C))
    _need_cuda(target, "target", torch.bfloat16, (B, L, C))
    _need_cuda(seq_id, "seq_id", torch.int32, (B, L))
    return B, L, C


def masked_mse_loss(pred, target, seq_id, grad: bool | torch.Tensor = False, grad_scale: float = 1.0,
                    loss=None, ws=None, stream=None):
    """Squared-error loss averaged over the valid tokens (seq_id >= 0), i.e.
    over the valid frames ("lingbot_va_packing" §2.1, compute_loss).  pred,
    target bf16 [B, L, C]; seq_id int32 [B, L].  Returns the fp32 loss as a
    one-element device tensor, or (loss, grad) when grad is True or a bf16
    [B, L, C] tensor to fill: grad = grad_scale * d loss / d pred, computed
    in the same pass."""
    B, L, C = _loss_args(pred, target, seq_id)
    want_grad = grad is not False and grad is not None
    g = None
    if want_grad:
        g = torch.empty_like(pred) if grad is True else grad
        _need_cuda(g, "grad", torch.bfloat16, (B, L, C))
    loss = torch.empty(1, dtype=torch.float32, device=pred.device) if loss is None else loss
    _need_cuda(loss, "loss", torch.float32, (1,))
    lib = _lib.load()
    nbytes = int(lib.masked_mse_ws_bytes(B, L, C))
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=pred.device)
    with torch.cuda.device(pred.device):
        _check(lib.masked_mse_loss(pred.data_ptr(), target.data_ptr(), seq_id.data_ptr(), B, L, C, loss.data_ptr(),
                                   _ptr(g), float(grad_scale), ws.data_ptr(), ws.numel(), _stream(stream)))
    return (loss, g) if want_grad else loss


def masked_mse_loss_bwd(pred, target, seq_id, dloss, grad=None, ws=None, stream=None):
    """d loss / d pred of masked_mse_loss times the device scalar dloss (fp32, one element)."""
    B, L, C = _loss_args(pred, target, seq_id)
    _need_cuda(dloss, "dloss", torch.float32)
    if dloss.numel() != 1:
        raise ValueError("dloss must hold one element")
    grad = torch.empty_like(pred) if grad is None else grad
    _need_cuda(grad, "grad", torch.bfloat16, (B, L, C))
    lib = _lib.load()
    nbytes = int(lib.masked_mse_ws_bytes(B, L, C))
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=pred.device)
    with torch.cuda.device(pred.device):
        _check(lib.masked_mse_loss_bwd(pred.data_ptr(), target.data_ptr(), seq_id.data_ptr(), B, L, C,
                                       dloss.data_ptr(), grad.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return grad


# ------------------------------------------------------------------- errors
def device_error(stream=None, raise_on_error: bool = True):
    """Synchronises the stream and returns (status, [code, where, block, thread])."""
    info = (ctypes.c_int32 * 4)()
    st = _lib.load().pvl_device_error_detail(_stream(stream), ctypes.addressof(info))
    msg = _lib.load().pvl_last_error_message().decode()
    if raise_on_error and st != PVL_OK:
        raise PvlError(st, msg)
    return st, list(info)


def set_attn_wait_timeout_ns(ns: int) -> None:
    """Bound on any single device-side wait of the attention kernels launched
    from now on, process-wide; 0 restores the default (2 s)."""
    _check(_lib.load().pvl_set_attn_wait_timeout_ns(int(ns)))


def _event_handle(ev) -> int | None:
    if ev is None:
        return None
    handle = int(ev.cuda_event)
    if handle == 0:
        raise ValueError("the event has no CUDA event yet: record it once before passing it")
    return handle


def mark_next_bwd_main(before, after) -> None:
    """Records the torch.cuda.Event objects ``before`` / ``after`` around the
    main backward kernel of this thread's next masked_attn_bwd call (one-shot;
    see pvl_mark_next_bwd_main).  Each event must have been recorded once
    already, so that its CUDA event exists."""
    _check(_lib.load().pvl_mark_next_bwd_main(_event_handle(before), _event_handle(after)))


def version() -> int:
    return int(_lib.load().pvl_version())
