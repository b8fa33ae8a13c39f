"""Python binding of the GB300 dense video-token attention library.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``_build/libfv.so`` (built from ``csrc/`` by ``build.py``), called through its
C ABI (``include/fv.h``) with ctypes.  torch supplies device memory and the
current stream.  There is no fallback: if the library is missing or the GPU
is not compute capability 10.3, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfv.so")
# the same library with the in-kernel index checks compiled in (FV_DEBUG_CHECKS=1)
DEBUG_LIB_PATH = os.path.join(_HERE, "_build", "libfv_debug.so")

STATUS = {
    0: "FV_OK", -1: "FV_ERR_NULL", -2: "FV_ERR_SHAPE", -3: "FV_ERR_ALIGN", -4: "FV_ERR_STEP",
    -5: "FV_ERR_UNSUPPORTED_DEVICE", -6: "FV_ERR_LAUNCH", -7: "FV_ERR_DEVICE_TIMEOUT", -8: "FV_ERR_ARG",
    -9: "FV_ERR_ALIAS", -10: "FV_ERR_DEVICE_CHECK",
}
# every symbol include/fv.h declares
EXPORTS = ("fv_attn_fwd", "fv_adaln_modulate", "fv_gated_residual", "fv_step_for_timestep", "fv_sync_status",
           "fv_status_string", "fv_version", "fv_attn_fwd_noalloc", "fv_attn_fwd_window",
           "fv_adaln_modulate_tagged", "fv_gated_residual_tagged", "fv_delta_attn", "fv_vsa_attn",
           "fv_vsa_num_tiles", "fv_vsa_topk", "fv_vsa_workspace_bytes", "fv_test_skip_load")
NOALLOC_MAX_LAUNCHES = 64

HEAD_DIM = 128
DEFAULT_SCALE = 1.0 / math.sqrt(HEAD_DIM)


class FvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libfv.so not built ({p}); run video_diffusion_transformer_gb300/build.py "
                          "or __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.fv_attn_fwd.argtypes = [vp, vp, vp, vp, i64, i32, i32, f32, i32, vp, vp]
    lib.fv_attn_fwd.restype = i32
    lib.fv_attn_fwd_window.argtypes = [vp, vp, vp, vp, i64, i32, i32, f32, i32, i32, i32, i32, vp, vp]
    lib.fv_attn_fwd_window.restype = i32
    lib.fv_delta_attn.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.fv_delta_attn.restype = i32
    lib.fv_vsa_attn.argtypes = [vp, vp, vp, vp, i64, i32, i32, f32, i32, i32, i32, i32, vp, vp, i64, vp, vp]
    lib.fv_vsa_attn.restype = i32
    lib.fv_vsa_num_tiles.argtypes = [i32, i32, i32]
    lib.fv_vsa_num_tiles.restype = i32
    lib.fv_vsa_topk.argtypes = [i32, ctypes.c_double]
    lib.fv_vsa_topk.restype = i32
    lib.fv_vsa_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.fv_vsa_workspace_bytes.restype = i64
    lib.fv_adaln_modulate.argtypes = [vp, vp, i32, i64, i32, vp, vp, i64, i32, i32, f32, vp]
    lib.fv_adaln_modulate.restype = i32
    lib.fv_gated_residual.argtypes = [vp, vp, vp, i64, i32, vp, i64, i32, i32, vp]
    lib.fv_gated_residual.restype = i32
    lib.fv_adaln_modulate_tagged.argtypes = [vp, vp, i32, i64, i32, vp, vp, i64, i32, i32, i32, vp, f32, vp]
    lib.fv_adaln_modulate_tagged.restype = i32
    lib.fv_gated_residual_tagged.argtypes = [vp, vp, vp, i64, i32, vp, i64, i32, i32, i32, vp, vp]
    lib.fv_gated_residual_tagged.restype = i32
    lib.fv_step_for_timestep.argtypes = [ctypes.POINTER(ctypes.c_float), i32, f32, ctypes.POINTER(ctypes.c_int)]
    lib.fv_step_for_timestep.restype = i32
    lib.fv_sync_status.argtypes = [vp]
    lib.fv_sync_status.restype = i32
    lib.fv_status_string.argtypes = [i32]
    lib.fv_status_string.restype = ctypes.c_char_p
    lib.fv_version.argtypes = []
    lib.fv_version.restype = i32
    lib.fv_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, i64, i32, i32, f32, i32, vp, vp, ctypes.POINTER(ctypes.c_int)]
    lib.fv_attn_fwd_noalloc.restype = i32
    lib.fv_test_skip_load.argtypes = [i32, i64]
    lib.fv_test_skip_load.restype = i32
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load_library().fv_status_string(int(code)).decode()
    except ImportError:
        return STATUS.get(int(code), f"status {code}")


def _check(code: int, where: str):
    if code != 0:
        raise FvError(code, where)


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None, *,
             heads: int | None = None, head_group: int = 16, scale: float = DEFAULT_SCALE,
             lse: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """O = softmax(Q K^T * scale) V per head, no mask.

    q, k, v: bf16 CUDA [N, H*128] (token-major) or [N, H, 128]; returns O of the
    same shape.  lse: optional float32 [H, N] filled with the log-sum-exp.
    """
    n = q.shape[0]
    width = q.numel() // max(1, n)
    h = heads if heads is not None else width // HEAD_DIM
    if h * HEAD_DIM != width or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [N, H*128]")
    if out is None:
        out = torch.empty_like(q)
    ptrs = [_dev(t, nm, torch.bfloat16) for t, nm in ((q, "q"), (k, "k"), (v, "v"), (out, "out"))]
    lse_ptr = None
    if lse is not None:
        if lse.shape != (h, n):
            raise ValueError("lse must be float32 [H, N]")
        lse_ptr = _dev(lse, "lse", torch.float32)
    code = load_library().fv_attn_fwd(*ptrs, n, h, HEAD_DIM, float(scale), int(min(head_group, h)), lse_ptr,
                                      _stream_ptr(stream))
    _check(code, "fv_attn_fwd")
    return out


def attn_fwd_window(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None, *,
                    frame_tokens: int, chunk_frames: int = 5, window_chunks: int = 1, heads: int | None = None,
                    head_group: int = 16, scale: float = DEFAULT_SCALE, lse: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Windowed softmax attention (the Video DeltaNet softmax branch): queries see
    keys in latent-frame chunks within ``window_chunks`` of their own, plus the
    first and last frame; queries in those two frames see every key."""
    n = q.shape[0]
    width = q.numel() // max(1, n)
    h = heads if heads is not None else width // HEAD_DIM
    if h * HEAD_DIM != width or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [N, H*128]")
    if out is None:
        out = torch.empty_like(q)
    ptrs = [_dev(t, nm, torch.bfloat16) for t, nm in ((q, "q"), (k, "k"), (v, "v"), (out, "out"))]
    lse_ptr = None
    if lse is not None:
        if lse.shape != (h, n):
            raise ValueError("lse must be float32 [H, N]")
        lse_ptr = _dev(lse, "lse", torch.float32)
    code = load_library().fv_attn_fwd_window(*ptrs, n, h, HEAD_DIM, float(scale), int(min(head_group, h)),
                                             int(frame_tokens), int(chunk_frames), int(window_chunks), lse_ptr,
                                             _stream_ptr(stream))
    _check(code, "fv_attn_fwd_window")
    return out


def delta_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor, alpha: torch.Tensor, *,
               frame_tokens: int, chunk_frames: int = 5, window_chunks: int = 1,
               text_state: torch.Tensor | None = None, out: torch.Tensor | None = None,
               states: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
               stream=None):
    """Video Delta Attention (the Video DeltaNet linear branch).

    q, k, v: bf16 [N, H*128]; beta: float32 [H, N]; alpha: float32 [H, F, 128];
    text_state: float32 [H, 128, 128] or None.  Returns (O bf16 [N, H*128],
    states float32 [2, H, F, 128, 128]).  ``workspace`` (float32, same shape as
    states) may be passed to avoid an allocation per call.
    """
    n = q.shape[0]
    h = (q.numel() // max(1, n)) // HEAD_DIM
    frames = n // frame_tokens
    if k.shape != q.shape or v.shape != q.shape or beta.shape != (h, n) or alpha.shape != (h, frames, HEAD_DIM):
        raise ValueError("shapes: q, k, v [N, H*128]; beta [H, N]; alpha [H, F, 128]")
    shape = (2, h, frames, HEAD_DIM, HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    if states is None:
        states = torch.empty(shape, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(shape, dtype=torch.float32, device=q.device)
    if states.shape != shape or workspace.shape != shape:
        raise ValueError("states and workspace must be float32 [2, H, F, 128, 128]")
    ts = None
    if text_state is not None:
        if text_state.shape != (h, HEAD_DIM, HEAD_DIM):
            raise ValueError("text_state must be float32 [H, 128, 128]")
        ts = _dev(text_state, "text_state", torch.float32)
    code = load_library().fv_delta_attn(
        _dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16),
        _dev(beta, "beta", torch.float32), _dev(alpha, "alpha", torch.float32), ts, n, h, HEAD_DIM,
        int(frame_tokens), int(chunk_frames), int(window_chunks), _dev(out, "out", torch.bfloat16),
        _dev(states, "states", torch.float32), _dev(workspace, "workspace", torch.float32), _stream_ptr(stream))
    _check(code, "fv_delta_attn")
    return out, states


def vsa_num_tiles(frames: int, height: int, width: int) -> int:
    """Tiles of the (4, 4, 4) tiling of a latent grid (fv_vsa_num_tiles)."""
    return int(load_library().fv_vsa_num_tiles(int(frames), int(height), int(width)))


def vsa_topk(num_tiles: int, sparsity: float) -> int:
    """Kept key tiles per query tile for a sparsity (fv_vsa_topk)."""
    return int(load_library().fv_vsa_topk(int(num_tiles), float(sparsity)))


def vsa_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, frames: int, height: int, width: int,
             topk: int | None = None, sparsity: float = 0.9, scale: float = DEFAULT_SCALE,
             out: torch.Tensor | None = None, selected: torch.Tensor | None = None,
             workspace: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """VSA-style block-sparse attention over a (frames, height, width) latent grid.

    q, k, v: bf16 [N, H*128] with N = frames*height*width in raster order.
    ``topk`` (default: the count for ``sparsity``) key tiles are kept per
    query tile.  Returns (O bf16 [N, H*128], selected int32 [H, tiles, topk]).
    ``workspace`` (uint8, at least fv_vsa_workspace_bytes) avoids an
    allocation per call.
    """
    lib = load_library()
    n = q.shape[0]
    width_all = q.numel() // max(1, n)
    h = width_all // HEAD_DIM
    if h * HEAD_DIM != width_all or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [N, H*128]")
    nt = vsa_num_tiles(frames, height, width)
    if nt < 1:
        raise ValueError("bad latent grid")
    if topk is None:
        topk = vsa_topk(nt, sparsity)
    if out is None:
        out = torch.empty_like(q)
    if selected is None:
        selected = torch.empty((h, nt, topk), dtype=torch.int32, device=q.device)
    if selected.shape != (h, nt, topk):
        raise ValueError("selected must be int32 [H, tiles, topk]")
    need = int(lib.fv_vsa_workspace_bytes(h, int(frames), int(height), int(width), int(topk)))
    if need < 0:
        raise FvError(-2, "fv_vsa_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lse_ptr = None
    if lse is not None:
        if lse.shape != (h, n):
            raise ValueError("lse must be float32 [H, N]")
        lse_ptr = _dev(lse, "lse", torch.float32)
    code = lib.fv_vsa_attn(_dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16),
                           _dev(out, "out", torch.bfloat16), n, h, HEAD_DIM, float(scale), int(frames), int(height),
                           int(width), int(topk), _dev(selected, "selected", torch.int32),
                           _dev(workspace, "workspace", torch.uint8), workspace.numel(), lse_ptr,
                           _stream_ptr(stream))
    _check(code, "fv_vsa_attn")
    return out, selected


def attn_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None, *,
                     heads: int | None = None, head_group: int = 16, scale: float = DEFAULT_SCALE,
                     lse: torch.Tensor | None = None, stream=None, check_device_status: bool = True) -> torch.Tensor:
    """attn_fwd without any device allocation by the library (fv_attn_fwd_noalloc).

    For callers whose device memory belongs to a pool they manage: the
    library's scratch lives in a fixed array compiled into it.  At most
    NOALLOC_MAX_LAUNCHES head-group launches per call.  With
    check_device_status the call waits for the stream and raises on a
    device-side timeout.
    """
    n = q.shape[0]
    width = q.numel() // max(1, n)
    h = heads if heads is not None else width // HEAD_DIM
    if h * HEAD_DIM != width or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [N, H*128]")
    if out is None:
        out = torch.empty_like(q)
    ptrs = [_dev(t, nm, torch.bfloat16) for t, nm in ((q, "q"), (k, "k"), (v, "v"), (out, "out"))]
    lse_ptr = None
    if lse is not None:
        if lse.shape != (h, n):
            raise ValueError("lse must be float32 [H, N]")
        lse_ptr = _dev(lse, "lse", torch.float32)
    dev_status = ctypes.c_int(0)
    code = load_library().fv_attn_fwd_noalloc(*ptrs, n, h, HEAD_DIM, float(scale), int(min(head_group, h)), lse_ptr,
                                              _stream_ptr(stream),
                                              ctypes.byref(dev_status) if check_device_status else None)
    _check(code, "fv_attn_fwd_noalloc")
    _check(dev_status.value, "fv_attn_fwd_noalloc (device)")
    return out


def adaln_modulate(x: torch.Tensor, shift_table: torch.Tensor, scale_table: torch.Tensor, step: int, *,
                   eps: float = 1e-6, out: torch.Tensor | None = None, out_dtype=torch.bfloat16,
                   stream=None) -> torch.Tensor:
    """y = LN(x) * (1 + scale_table[step]) + shift_table[step]; x bf16 [N, C], tables float32 [steps, C]."""
    n, c = x.shape
    if out is None:
        out = torch.empty((n, c), dtype=out_dtype, device=x.device)
    if shift_table.shape != scale_table.shape or shift_table.dim() != 2:
        raise ValueError("tables must be float32 [steps, ld]")
    for t, nm in ((shift_table, "shift_table"), (scale_table, "scale_table")):
        if t.stride(1) != 1:
            raise ValueError(f"{nm} rows must be contiguous")
    if out.dtype not in (torch.bfloat16, torch.float32) or out.shape != (n, c):
        raise ValueError("out must be bfloat16 or float32 [N, C]")
    code = load_library().fv_adaln_modulate(
        _dev(x, "x", torch.bfloat16), _dev(out, "out", out.dtype), 1 if out.dtype == torch.float32 else 0, n, c,
        shift_table.data_ptr(), scale_table.data_ptr(), shift_table.stride(0), shift_table.shape[0], int(step),
        float(eps), _stream_ptr(stream))
    _check(code, "fv_adaln_modulate")
    return out


def gated_residual(x: torch.Tensor, a: torch.Tensor, gate_table: torch.Tensor, step: int, *,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out = x + gate_table[step] * a (bf16 [N, C]); out may be x itself."""
    n, c = x.shape
    if out is None:
        out = torch.empty_like(x)
    if gate_table.dim() != 2 or gate_table.stride(1) != 1:
        raise ValueError("gate_table must be float32 [steps, ld] with contiguous rows")
    code = load_library().fv_gated_residual(
        _dev(x, "x", torch.bfloat16), _dev(a, "a", torch.bfloat16), _dev(out, "out", torch.bfloat16), n, c,
        gate_table.data_ptr(), gate_table.stride(0), gate_table.shape[0], int(step), _stream_ptr(stream))
    _check(code, "fv_gated_residual")
    return out


def adaln_modulate_tagged(x: torch.Tensor, shift_table: torch.Tensor, scale_table: torch.Tensor, step: int,
                          tags: torch.Tensor, num_modalities: int, *, eps: float = 1e-6,
                          out: torch.Tensor | None = None, out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """Modulate with per-token modality rows: token i reads table row
    step * num_modalities + tags[i] (tables float32 [steps * num_modalities, C])."""
    n, c = x.shape
    if out is None:
        out = torch.empty((n, c), dtype=out_dtype, device=x.device)
    if shift_table.shape != scale_table.shape or shift_table.dim() != 2 or shift_table.stride(1) != 1 \
            or scale_table.stride(1) != 1:
        raise ValueError("tables must be float32 [steps * modalities, ld] with contiguous rows")
    if shift_table.shape[0] % num_modalities:
        raise ValueError("table rows must be steps * num_modalities")
    if tags.shape != (n,):
        raise ValueError("tags must be uint8 [N]")
    code = load_library().fv_adaln_modulate_tagged(
        _dev(x, "x", torch.bfloat16), _dev(out, "out", out.dtype), 1 if out.dtype == torch.float32 else 0, n, c,
        shift_table.data_ptr(), scale_table.data_ptr(), shift_table.stride(0), shift_table.shape[0] // num_modalities,
        int(num_modalities), int(step), _dev(tags, "tags", torch.uint8), float(eps), _stream_ptr(stream))
    _check(code, "fv_adaln_modulate_tagged")
    return out


def gated_residual_tagged(x: torch.Tensor, a: torch.Tensor, gate_table: torch.Tensor, step: int,
                          tags: torch.Tensor, num_modalities: int, *, out: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """Gated residual with per-token modality rows of the gate table."""
    n, c = x.shape
    if out is None:
        out = torch.empty_like(x)
    if gate_table.dim() != 2 or gate_table.stride(1) != 1 or gate_table.shape[0] % num_modalities:
        raise ValueError("gate_table must be float32 [steps * modalities, ld] with contiguous rows")
    if tags.shape != (n,):
        raise ValueError("tags must be uint8 [N]")
    code = load_library().fv_gated_residual_tagged(
        _dev(x, "x", torch.bfloat16), _dev(a, "a", torch.bfloat16), _dev(out, "out", torch.bfloat16), n, c,
        gate_table.data_ptr(), gate_table.stride(0), gate_table.shape[0] // num_modalities, int(num_modalities),
        int(step), _dev(tags, "tags", torch.uint8), _stream_ptr(stream))
    _check(code, "fv_gated_residual_tagged")
    return out


def step_for_timestep(ladder, t: float) -> int:
    """Index of timestep t on the stored ladder; raises FvError(FV_ERR_STEP) if absent."""
    arr = (ctypes.c_float * len(ladder))(*[float(v) for v in ladder])
    out = ctypes.c_int(-1)
    _check(load_library().fv_step_for_timestep(arr, len(ladder), float(t), ctypes.byref(out)),
           "fv_step_for_timestep")
    return out.value


# fv_test_kernel values (include/fv.h)
TEST_ATTN, TEST_VSA_FINE, TEST_VDA_STATS, TEST_VDA_SCAN, TEST_VDA_READOUT = range(5)


def test_skip_load(kernel: int, load_index: int) -> None:
    """Test hook (fv_test_skip_load): the next launch of ``kernel`` has its
    first CTA never issue copy number ``load_index``, so a bounded wait runs
    out and the call reports FV_ERR_DEVICE_TIMEOUT.  One-shot; a negative
    index disarms it."""
    _check(load_library().fv_test_skip_load(int(kernel), int(load_index)), "fv_test_skip_load")


def sync_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a device-side error."""
    _check(load_library().fv_sync_status(_stream_ptr(stream)), "fv_sync_status")
