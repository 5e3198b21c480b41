"""Python binding of libdflash.so (DFlash draft body + greedy verification on GB300).

Argument marshalling only: every function here converts torch tensors to device pointers
and sizes, calls the C ABI function of the same name, and raises on a non-OK status
(ValueError for DFLASH_ERR_INVALID_ARG, RuntimeError otherwise).  All compute happens in
the library's CUDA kernels.  There is no fallback: if the library has not been built the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libdflash.so")
INCLUDE_DIR = os.path.join(os.path.dirname(HERE), "include")

DFLASH_OK = 0
DFLASH_ERR_INVALID_ARG = 1
DFLASH_ERR_UNSUPPORTED = 2
DFLASH_ERR_CUDA = 3
DFLASH_ERR_TIMEOUT = 4
DFLASH_ERR_DEVICE_CHECK = 5
DFLASH_ERR_RANGE = 6
DFLASH_DTYPE_F32 = 0
DFLASH_DTYPE_BF16 = 1
DFLASH_DTYPE_F16 = 2
DFLASH_FLAG_FINAL_NORM = 1
DFLASH_FLAG_CTX_NORM = 2
DFLASH_FLAG_F16_LAYERS = 4
DFLASH_TESTING_ENGINE_TC = 0
DFLASH_TESTING_ENGINE_SIMT = 1
PROF_KINDS = {"gemm": 0, "attention": 1, "rows": 2, "plan": 3, "verify": 4, "convert": 5}
LAYER_MATRICES = ("w_qkv", "w_o", "w_gate_up", "w_down")


class dflash_config_t(ctypes.Structure):
    _fields_ = [("target_hidden", ctypes.c_int32), ("num_target_layers", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double)]


class dflash_layer_weights_t(ctypes.Structure):
    _fields_ = [("g_in", ctypes.c_void_p), ("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("g_post", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p)]


class dflash_weights_t(ctypes.Structure):
    _fields_ = [("w_proj", ctypes.c_void_p), ("g_ctx", ctypes.c_void_p),
                ("g_final", ctypes.c_void_p),
                ("layers", ctypes.POINTER(dflash_layer_weights_t)),
                ("num_layers", ctypes.c_int32)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_long
_Z = ctypes.c_size_t
_SIGS = {
    "dflash_last_error": (ctypes.c_char_p, []),
    "dflash_version": (_I, []),
    "dflash_device_status": (_I, [_I]),
    "dflash_convert_bf16_to_f16": (_I, [_P, _P, _Z, _P]),
    "dflash_plan_workspace_size": (_Z, [_I, _I, _I, _I]),
    "dflash_plan": (_I, [_P, _P, _I, _I, ctypes.c_int64, ctypes.c_uint64, _I, _I, _P, _P, _P, _P,
                         _P, _P, _Z, _P]),
    "dflash_project_context_workspace_size": (_Z, [ctypes.POINTER(dflash_config_t), _I, _I]),
    "dflash_project_context": (_I, [ctypes.POINTER(dflash_config_t),
                                    ctypes.POINTER(dflash_weights_t), _P, _I, _I, _I, _I, _P, _P,
                                    _P, _Z, _P]),
    "dflash_append_context_workspace_size": (_Z, [ctypes.POINTER(dflash_config_t), _I, _I, _I]),
    "dflash_append_context": (_I, [ctypes.POINTER(dflash_config_t),
                                   ctypes.POINTER(dflash_weights_t), _P, _I, _I, _P, _P, _I, _P,
                                   _P, _Z, _P]),
    "dflash_body_workspace_size": (_Z, [ctypes.POINTER(dflash_config_t), _I, _I, _I]),
    "dflash_body_forward": (_I, [ctypes.POINTER(dflash_config_t), ctypes.POINTER(dflash_weights_t),
                                 _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _Z, _P]),
    "dflash_decayed_ce_workspace_size": (_Z, [_I, _I, _I]),
    "dflash_decayed_ce_loss": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_double, _P, _P, _P,
                                    _Z, _P]),
    "dflash_verify_workspace_size": (_Z, [_I, _I, _I]),
    "dflash_verify_greedy": (_I, [_P, _I, _P, _I, _I, _I, ctypes.c_int32, _P, _P, _P, _P, _P, _Z,
                                  _P]),
    "dflash_verify_sampling_workspace_size": (_Z, [_I, _I, _I]),
    "dflash_verify_sampling": (_I, [_P, _I, ctypes.c_double, _P, _P, _I, _I, _I, ctypes.c_uint64,
                                    ctypes.c_int32, _P, _P, _P, _P, _Z, _P]),
    "dflash_verify_greedy_static": (_I, [_P, _I, _P, _I, _I, _I, ctypes.c_int32, _P, _P, _P, _P,
                                         _P]),
    "dflash_testing_gemm": (_I, [_I, _I, _P, _L, _P, _L, _P, _L, _L, _I, _I, _I, _P]),
    "dflash_testing_gemm_splits": (_I, [_L, _I, _I]),
    "dflash_testing_fused_epilogues": (_I, [_I]),
    "dflash_testing_gemm_pairs": (_I, [_I]),
    "dflash_testing_rope_table": (_I, [_P, _P, _I, _I, _I, ctypes.c_double, _P]),
    "dflash_testing_gemm_withheld": (_I, [_P, _L, _P, _L, _P, _L, _L, _I, _I, _L, _P]),
    "dflash_testing_gemm_ws": (_I, [_P, _L, _P, _I, _L, _P, _L, _L, _I, _I, _I, _P, _P, _P]),
    "dflash_testing_verify_plan": (_I, [_I, _I, _I, _L, _L, ctypes.POINTER(_I),
                                       ctypes.POINTER(_I)]),
    "dflash_profile_enable": (_I, [_I]),
    "dflash_profile_read": (_I, [_I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_L)]),
    "dflash_launch_count": (_L, []),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libdflash.so (built in-tree by build.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdflash.so is not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def declared_symbols() -> list:
    """Every function declared in include/*.h."""
    names = []
    for fn in sorted(os.listdir(INCLUDE_DIR)):
        if fn.endswith(".h"):
            with open(os.path.join(INCLUDE_DIR, fn)) as f:
                names += re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", f.read())
    return names


def _check(status: int) -> None:
    if status == DFLASH_OK:
        return
    msg = load().dflash_last_error().decode(errors="replace")
    if status == DFLASH_ERR_INVALID_ARG:
        raise ValueError(msg)
    raise RuntimeError(f"dflash status {status}: {msg}")


# ---- helpers ------------------------------------------------------------------------------

def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def make_config(shape, f16_layers: bool = False) -> dflash_config_t:
    """dflash_config_t from any object with the DFlash shape fields (see dflash_inputs);
    f16_layers sets DFLASH_FLAG_F16_LAYERS (weights from prepare_f16_layers)."""
    return dflash_config_t(
        target_hidden=shape.target_hidden, num_target_layers=shape.num_target_layers,
        hidden=shape.hidden, num_layers=shape.num_layers, num_heads=shape.num_heads,
        num_kv_heads=shape.num_kv_heads, head_dim=shape.head_dim,
        intermediate=shape.intermediate, block_size=shape.block_size,
        dtype=DFLASH_DTYPE_BF16 if shape.dtype == "bf16" else DFLASH_DTYPE_F32,
        flags=(DFLASH_FLAG_FINAL_NORM if shape.final_norm else 0) |
              (DFLASH_FLAG_CTX_NORM if shape.ctx_norm else 0) |
              (DFLASH_FLAG_F16_LAYERS if f16_layers else 0),
        reserved=0, rope_theta=float(shape.rope_theta), rms_eps=float(shape.rms_eps))


class Weights:
    """Keeps the ctypes weight structs (and the tensors they point to) alive."""

    def __init__(self, top: dict, layers: list):
        self.tensors = (top, layers)
        arr = (dflash_layer_weights_t * len(layers))()
        for i, lw in enumerate(layers):
            arr[i] = dflash_layer_weights_t(*(lw[k].data_ptr() for k in
                                              ("g_in", "w_qkv", "w_o", "g_post", "w_gate_up",
                                               "w_down")))
        self._layers = arr
        self.struct = dflash_weights_t(top["w_proj"].data_ptr(), top["g_ctx"].data_ptr(),
                                       top["g_final"].data_ptr(), arr, len(layers))


def dflash_convert_bf16_to_f16(src, dst, stream=None) -> None:
    if dst.numel() != src.numel():
        raise ValueError("dst must have as many elements as src")
    _check(load().dflash_convert_bf16_to_f16(_ptr(src), _ptr(dst), src.numel(), _stream(stream)))


def prepare_f16_layers(weights: Weights, out: list | None = None, stream=None) -> Weights:
    """Weights whose layer matrices are fp16 copies (dflash_convert_bf16_to_f16) of the bf16
    ones, for a config made with f16_layers=True.  `out` (optional) is a list of per-layer
    dicts of preallocated fp16 tensors to fill, reused across weight updates."""
    import torch
    top, layers = weights.tensors
    new_layers = []
    for i, lw in enumerate(layers):
        nl = dict(lw)
        for k in LAYER_MATRICES:
            dst = out[i][k] if out is not None else torch.empty(lw[k].shape, dtype=torch.float16,
                                                                 device=lw[k].device)
            dflash_convert_bf16_to_f16(lw[k], dst, stream)
            nl[k] = dst
        new_layers.append(nl)
    return Weights(top, new_layers)


def kv_cache_dtype(cfg):
    """torch dtype of the context K/V cache planes for a config: fp16 in the bf16
    configuration, fp32 in the fp32 one."""
    import torch
    return torch.float16 if cfg.dtype == DFLASH_DTYPE_BF16 else torch.float32


def workspace(nbytes: int, device="cuda"):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---- the four operations ---------------------------------------------------------------------

def dflash_plan(mask, sample_ids, step, seed, num_anchors, block_size, anchors, block_valid,
                loss_mask, position_ids, ctx_len=None, ws=None, stream=None):
    lib = load()
    B, L = mask.shape
    need = lib.dflash_plan_workspace_size(B, L, num_anchors, block_size)
    ws = ws if ws is not None else (workspace(need, mask.device) if need else None)
    _check(lib.dflash_plan(_ptr(mask), _ptr(sample_ids), B, L, int(step),
                           int(seed) & ((1 << 64) - 1), num_anchors, block_size, _ptr(anchors),
                           _ptr(block_valid), _ptr(loss_mask), _ptr(position_ids),
                           _ptr(ctx_len), _ptr(ws), 0 if ws is None else ws.numel(),
                           _stream(stream)))


def dflash_project_context_workspace_size(cfg, B, L) -> int:
    return load().dflash_project_context_workspace_size(ctypes.byref(cfg), B, L)


def dflash_project_context(cfg, weights, target_hidden, B, L, pos_offset, L_cache, kv_cache,
                           ctx_len=None, ws=None, stream=None):
    lib = load()
    if ws is None:
        ws = workspace(dflash_project_context_workspace_size(cfg, B, L), target_hidden.device)
    _check(lib.dflash_project_context(ctypes.byref(cfg), ctypes.byref(weights.struct),
                                      _ptr(target_hidden), B, L, pos_offset, L_cache,
                                      _ptr(ctx_len), _ptr(kv_cache), _ptr(ws), ws.numel(),
                                      _stream(stream)))


def dflash_append_context_workspace_size(cfg, B, P, L_cache) -> int:
    return load().dflash_append_context_workspace_size(ctypes.byref(cfg), B, P, L_cache)


def dflash_append_context(cfg, weights, target_hidden, B, P, accepted, cache_len, L_cache,
                          kv_cache, ws=None, stream=None):
    lib = load()
    if ws is None:
        ws = workspace(dflash_append_context_workspace_size(cfg, B, P, L_cache),
                       target_hidden.device)
    _check(lib.dflash_append_context(ctypes.byref(cfg), ctypes.byref(weights.struct),
                                     _ptr(target_hidden), B, P, _ptr(accepted), _ptr(cache_len),
                                     L_cache, _ptr(kv_cache), _ptr(ws), ws.numel(),
                                     _stream(stream)))


def dflash_body_workspace_size(cfg, B, L, N) -> int:
    return load().dflash_body_workspace_size(ctypes.byref(cfg), B, L, N)


def dflash_body_forward(cfg, weights, block_emb, anchors, block_valid, position_ids, mask,
                        kv_cache, B, L, N, out, ws=None, stream=None):
    lib = load()
    if ws is None:
        ws = workspace(dflash_body_workspace_size(cfg, B, L, N), block_emb.device)
    _check(lib.dflash_body_forward(ctypes.byref(cfg), ctypes.byref(weights.struct),
                                   _ptr(block_emb), _ptr(anchors), _ptr(block_valid),
                                   _ptr(position_ids), _ptr(mask), _ptr(kv_cache), B, L, N,
                                   _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def dflash_decayed_ce_loss(hidden, lm_head, targets, loss_mask, T, block_size, D, V, decay, ce,
                           loss, ws=None, stream=None):
    lib = load()
    if ws is None:
        ws = workspace(lib.dflash_decayed_ce_workspace_size(T, D, V), hidden.device)
    _check(lib.dflash_decayed_ce_loss(_ptr(hidden), _ptr(lm_head), _ptr(targets),
                                      _ptr(loss_mask), T, block_size, D, V, float(decay), _ptr(ce),
                                      _ptr(loss), _ptr(ws), ws.numel(), _stream(stream)))


def dflash_verify_workspace_size(B, gamma, V) -> int:
    return load().dflash_verify_workspace_size(B, gamma, V)


def dflash_verify_greedy(logits, logits_dtype, draft, B, gamma, V, eos, emitted, num_emitted,
                         accepted, target_choices=None, ws=None, stream=None):
    lib = load()
    if ws is None:
        ws = workspace(dflash_verify_workspace_size(B, gamma, V), logits.device)
    _check(lib.dflash_verify_greedy(_ptr(logits), logits_dtype, _ptr(draft), B, gamma, V,
                                    int(eos), _ptr(emitted), _ptr(num_emitted), _ptr(accepted),
                                    _ptr(target_choices), _ptr(ws), ws.numel(), _stream(stream)))


def dflash_verify_sampling(logits, logits_dtype, temperature, draft_probs, draft, B, gamma, V,
                           seed, eos, emitted, num_emitted, accepted, ws=None, stream=None):
    lib = load()
    if ws is None:
        ws = workspace(lib.dflash_verify_sampling_workspace_size(B, gamma, V), logits.device)
    _check(lib.dflash_verify_sampling(_ptr(logits), logits_dtype, float(temperature),
                                      _ptr(draft_probs), _ptr(draft), B, gamma, V,
                                      int(seed) & ((1 << 64) - 1), int(eos), _ptr(emitted),
                                      _ptr(num_emitted), _ptr(accepted), _ptr(ws), ws.numel(),
                                      _stream(stream)))


def dflash_verify_greedy_static(logits, logits_dtype, draft, B, gamma, V, eos, emitted,
                                num_emitted, accepted, target_choices=None, stream=None):
    """Greedy verification that allocates nothing (fixed scratch inside the library)."""
    _check(load().dflash_verify_greedy_static(_ptr(logits), logits_dtype, _ptr(draft), B, gamma,
                                              V, int(eos), _ptr(emitted), _ptr(num_emitted),
                                              _ptr(accepted), _ptr(target_choices),
                                              _stream(stream)))


def dflash_device_status(reset: bool = True) -> None:
    _check(load().dflash_device_status(1 if reset else 0))


def dflash_testing_gemm(engine, dtype, A, B, C, splits=1, stream=None):
    M, K = A.shape
    N = B.shape[0]
    _check(load().dflash_testing_gemm(engine, dtype, _ptr(A), A.stride(0), _ptr(B), B.stride(0),
                                      _ptr(C), C.stride(-2), M, N, K, splits, _stream(stream)))


def dflash_testing_gemm_withheld(A, B, C, wait_ns, stream=None):
    M, K = A.shape
    N = B.shape[0]
    _check(load().dflash_testing_gemm_withheld(_ptr(A), A.stride(0), _ptr(B), B.stride(0), _ptr(C),
                                               C.stride(-2), M, N, K, int(wait_ns),
                                               _stream(stream)))


def dflash_testing_gemm_ws(X, W, w_dtype, C, max_splits, splits_out, tile_list=None,
                           stream=None):
    M, K = X.shape
    N = W.shape[0]
    _check(load().dflash_testing_gemm_ws(_ptr(X), X.stride(0), _ptr(W), w_dtype, W.stride(0),
                                         _ptr(C), C.stride(-2), M, N, K, max_splits,
                                         _ptr(tile_list), _ptr(splits_out), _stream(stream)))


def dflash_testing_gemm_pairs(mode: int) -> None:
    """0: the 128 x 256-tile GEMM runs as CTA pairs from two M tiles up (default); 1: one
    CTA per tile everywhere."""
    _check(load().dflash_testing_gemm_pairs(mode))


def dflash_testing_rope_table(cos_t, sin_t, p0: int, head_dim: int, theta: float,
                              stream=None) -> None:
    """The device RoPE table: cos_t / sin_t float32 [P, head_dim / 2] for positions p0 .. p0+P-1."""
    P = cos_t.shape[0]
    _check(load().dflash_testing_rope_table(_ptr(cos_t), _ptr(sin_t), p0, P, head_dim, theta,
                                            _stream(stream)))


def dflash_testing_fused_epilogues(mode: int) -> None:
    """0: fused QKV / residual epilogues where no K-split is needed (default); 1: on every
    call on the 128 x 256-tile GEMM; 2: never."""
    _check(load().dflash_testing_fused_epilogues(mode))


def dflash_testing_verify_plan(B, gamma, V, resident_ctas, static_entries=0) -> tuple:
    """(chunks, chunk_len) of the verification argmax for these sizes (host arithmetic)."""
    c, n = ctypes.c_int(), ctypes.c_int()
    _check(load().dflash_testing_verify_plan(B, gamma, V, resident_ctas, static_entries,
                                             ctypes.byref(c), ctypes.byref(n)))
    return c.value, n.value


def dflash_profile_enable(on: bool = True) -> None:
    _check(load().dflash_profile_enable(1 if on else 0))


def dflash_profile_read() -> dict:
    """{kind: (total_ms, launches)} for every kernel kind recorded since enabling."""
    lib = load()
    out = {}
    for name, kind in PROF_KINDS.items():
        ms, n = ctypes.c_double(), ctypes.c_long()
        _check(lib.dflash_profile_read(kind, ctypes.byref(ms), ctypes.byref(n)))
        out[name] = (ms.value, n.value)
    return out


def dflash_launch_count() -> int:
    return int(load().dflash_launch_count())
