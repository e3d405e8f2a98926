"""Python binding of libfpd — the GB300 (sm_103a) block-drafter hot path.

Argument marshalling only: every step of the path runs in the CUDA kernels of ``libfpd.so`` behind the
C ABI of ``include/fpd.h``.  The functions keep the C names (``fpd_prepare_context``, ``fpd_draft_block``,
``fpd_constrain_argmax``, ``fpd_verify`` ...) and take torch CUDA tensors (or raw device addresses) for
device arguments.  PyTorch only provides device memory and streams.

There is no fallback: importing works without the library, but every call raises ``RuntimeError`` when
``libfpd.so`` has not been built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# FPD_LIBRARY=debug selects the FPD_DEBUG build (every call waits for its kernels and reports their errors)
LIB_PATH = os.path.join(_HERE, "libfpd_debug.so" if os.environ.get("FPD_LIBRARY") == "debug" else "libfpd.so")
MAX_LAYERS = 8

FPD_OK = 0
STATUS = {0: "FPD_OK", 1: "FPD_ERR_INVALID_ARG", 2: "FPD_ERR_SHAPE", 3: "FPD_ERR_CAPACITY",
          4: "FPD_ERR_UNSUPPORTED", 5: "FPD_ERR_CUDA", 6: "FPD_ERR_DEVICE_CHECK"}
FPD_VERIFY_TEXT, FPD_VERIFY_SCHEMA = 0, 1
FPD_RULE_NONE, FPD_RULE_MEMBER, FPD_RULE_DIGIT, FPD_RULE_DIGIT_LAST, FPD_RULE_CONFIDENT = 0, 1, 2, 3, 4


class GridFormat(ctypes.Structure):
    _fields_ = [("digit_id", ctypes.c_int32 * 10), ("plus_id", ctypes.c_int32), ("minus_id", ctypes.c_int32),
                ("pad_id", ctypes.c_int32), ("n_axes", ctypes.c_int32), ("width", ctypes.c_int32),
                ("axis_sep", ctypes.c_char), ("point_sep", ctypes.c_char)]


class FpdError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {msg}")
        self.status = status


class ModelDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("n_feat", ctypes.c_int32), ("max_pos", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("w_fc", ctypes.c_void_p), ("hidden_norm", ctypes.c_void_p),
                ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)] + [
        (n, ctypes.c_void_p * MAX_LAYERS) for n in
        ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "mlp_norm", "w_gate_up", "w_down")]


class VocabLayout(ctypes.Structure):
    _fields_ = [("n_class", ctypes.c_int32), ("class_off", ctypes.POINTER(ctypes.c_int32)),
                ("class_ranges", ctypes.POINTER(ctypes.c_int32)), ("pos_class", ctypes.c_void_p),
                ("n_pairs", ctypes.c_int32), ("pairs", ctypes.POINTER(ctypes.c_int16)), ("off_id", ctypes.c_int32)]


_lib = None
_EXPORTS = ["fpd_model_create", "fpd_model_destroy", "fpd_kv_store_bytes", "fpd_workspace_bytes",
            "fpd_prepare_context", "fpd_prepare_context_rows", "fpd_draft_block", "fpd_constrain_argmax",
            "fpd_constrain_argmax_noalloc", "fpd_verify", "fpd_verify_prefix", "fpd_sd_advance", "fpd_grid_to_text",
            "fpd_model_enable_fp8", "fpd_model_fp8_enabled", "fpd_quantize_fp8", "fpd_last_error",
            "fpd_kernel_launches", "fpd_device_status"]


def lib():
    """Load libfpd.so (raises when it has not been built — there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libfpd.so not built at {LIB_PATH}; run __graft_entry__.build()")
        l = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        l.fpd_model_create.argtypes = [ctypes.POINTER(ModelDesc), ctypes.POINTER(Weights), ctypes.POINTER(vp)]
        l.fpd_model_destroy.argtypes = [vp]
        l.fpd_model_destroy.restype = None
        l.fpd_kv_store_bytes.argtypes = [vp, ctypes.c_int, ctypes.c_int]
        l.fpd_kv_store_bytes.restype = sz
        l.fpd_workspace_bytes.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        l.fpd_workspace_bytes.restype = sz
        l.fpd_prepare_context.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.POINTER(vp), vp,
                                          ctypes.c_int, vp, sz, vp]
        l.fpd_prepare_context_rows.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.POINTER(vp), vp,
                                               ctypes.c_int, vp, sz, vp]
        l.fpd_sd_advance.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp]
        l.fpd_verify_prefix.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_float, ctypes.POINTER(VocabLayout),
                                        vp, i32, vp, vp, vp, vp]
        l.fpd_grid_to_text.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, ctypes.POINTER(GridFormat), ctypes.c_char_p,
                                       sz, ctypes.POINTER(sz)]
        l.fpd_draft_block.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int, vp, vp, i32, vp, vp, vp,
                                      sz, vp]
        l.fpd_constrain_argmax.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.POINTER(VocabLayout), vp, vp,
                                           vp, vp, sz, vp]
        l.fpd_constrain_argmax_noalloc.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, ctypes.POINTER(VocabLayout),
                                                   vp, vp, vp]
        l.fpd_verify.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.POINTER(VocabLayout), vp,
                                 i32, vp, vp, vp, vp]
        l.fpd_last_error.restype = ctypes.c_char_p
        l.fpd_kernel_launches.restype = ctypes.c_uint64
        l.fpd_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        l.fpd_model_enable_fp8.argtypes = [vp, vp]
        l.fpd_model_fp8_enabled.argtypes = [vp]
        l.fpd_model_fp8_enabled.restype = ctypes.c_int32
        l.fpd_quantize_fp8.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        for f in ("fpd_model_create", "fpd_model_enable_fp8", "fpd_quantize_fp8", "fpd_prepare_context", "fpd_prepare_context_rows", "fpd_draft_block",
                  "fpd_constrain_argmax", "fpd_constrain_argmax_noalloc", "fpd_verify", "fpd_sd_advance",
                  "fpd_grid_to_text", "fpd_verify_prefix",
                  "fpd_device_status"):
            getattr(l, f).restype = ctypes.c_int
        _lib = l
    return _lib


def _check(status: int, where: str) -> None:
    if status != FPD_OK:
        raise FpdError(status, where, lib().fpd_last_error().decode())


def _ptr(t) -> int | None:
    """Device address of a torch tensor, an int address, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("device tensors passed to libfpd must be contiguous (row-major)")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- C entry points, same names ------------------------------------------------------------------------------

def fpd_model_create(desc: ModelDesc, weights: Weights) -> int:
    h = ctypes.c_void_p()
    _check(lib().fpd_model_create(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(h)), "fpd_model_create")
    return h.value


def fpd_model_destroy(model: int) -> None:
    lib().fpd_model_destroy(model)


def fpd_model_enable_fp8(model: int, stream=None) -> None:
    _check(lib().fpd_model_enable_fp8(model, _stream(stream)), "fpd_model_enable_fp8")


def fpd_model_fp8_enabled(model: int) -> bool:
    return bool(lib().fpd_model_fp8_enabled(model))


def fpd_quantize_fp8(w, rows, cols, ld, codes, exps, stream=None) -> None:
    _check(lib().fpd_quantize_fp8(_ptr(w), rows, cols, ld, _ptr(codes), _ptr(exps), _stream(stream)),
           "fpd_quantize_fp8")


def fpd_kv_store_bytes(model: int, batch: int, t_cap: int) -> int:
    return int(lib().fpd_kv_store_bytes(model, batch, t_cap))


def fpd_workspace_bytes(model: int, batch: int, max_block_len: int, t_cap: int) -> int:
    return int(lib().fpd_workspace_bytes(model, batch, max_block_len, t_cap))


def fpd_prepare_context(model, batch, total_rows, row_off, pos_start, feats, kv_store, t_cap, workspace,
                        workspace_bytes, stream=None):
    arr = (ctypes.c_void_p * len(feats))(*[_ptr(f) for f in feats])
    _check(lib().fpd_prepare_context(model, batch, total_rows, _ptr(row_off), _ptr(pos_start), arr, _ptr(kv_store),
                                     t_cap, _ptr(workspace), workspace_bytes, _stream(stream)), "fpd_prepare_context")


def fpd_prepare_context_rows(model, batch, total_rows, row_off, row_cnt, pos_start, feats, kv_store, t_cap, workspace,
                             workspace_bytes, stream=None):
    arr = (ctypes.c_void_p * len(feats))(*[_ptr(f) for f in feats])
    _check(lib().fpd_prepare_context_rows(model, batch, total_rows, _ptr(row_off), _ptr(row_cnt), _ptr(pos_start),
                                          arr, _ptr(kv_store), t_cap, _ptr(workspace), workspace_bytes,
                                          _stream(stream)), "fpd_prepare_context_rows")


def fpd_sd_advance(batch, block_len, t_cap, accept_len, committed, ctx_len, pos_start, anchor, stream=None):
    _check(lib().fpd_sd_advance(batch, block_len, t_cap, _ptr(accept_len), _ptr(committed), _ptr(ctx_len),
                                _ptr(pos_start), _ptr(anchor), _stream(stream)), "fpd_sd_advance")


def fpd_draft_block(model, batch, block_len, kv_store, t_cap, ctx_len, anchor, mask_id, hidden_out,
                    layer_hidden, workspace, workspace_bytes, stream=None):
    _check(lib().fpd_draft_block(model, batch, block_len, _ptr(kv_store), t_cap, _ptr(ctx_len), _ptr(anchor),
                                 int(mask_id), _ptr(hidden_out), _ptr(layer_hidden), _ptr(workspace),
                                 workspace_bytes, _stream(stream)), "fpd_draft_block")


def make_layout(class_off, class_ranges, pos_class_dev, pairs=None, off_id=0) -> VocabLayout:
    """Build an fpd_vocab_layout: class tables from host sequences, pos_class a device tensor (int16); pairs an
    optional host sequence of (p, q) block positions of the off-screen pairing rule with its off_id."""
    import numpy as np
    co = np.ascontiguousarray(class_off, dtype=np.int32)
    cr = np.ascontiguousarray(class_ranges, dtype=np.int32)
    pr = np.ascontiguousarray(np.zeros((0, 2)) if pairs is None else pairs, dtype=np.int16).reshape(-1)
    lay = VocabLayout(len(co) - 1, co.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                      cr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(pos_class_dev), len(pr) // 2,
                      pr.ctypes.data_as(ctypes.POINTER(ctypes.c_int16)) if len(pr) else None, int(off_id))
    lay._keep = (co, cr, pos_class_dev, pr)
    return lay


def fpd_constrain_argmax(model, batch, block_len, hidden, layout, tokens_out, logits_out, workspace,
                         workspace_bytes, stream=None, margin_out=None):
    _check(lib().fpd_constrain_argmax(model, batch, block_len, _ptr(hidden),
                                      ctypes.byref(layout) if layout is not None else None, _ptr(tokens_out),
                                      _ptr(logits_out), _ptr(margin_out), _ptr(workspace), workspace_bytes,
                                      _stream(stream)),
           "fpd_constrain_argmax")


def fpd_constrain_argmax_noalloc(model, batch, block_len, hidden, layout, tokens_out, logits_out, stream=None):
    """fpd_constrain_argmax for callers that cannot allocate: the scratch is the library's static device array."""
    _check(lib().fpd_constrain_argmax_noalloc(model, batch, block_len, _ptr(hidden),
                                              ctypes.byref(layout) if layout is not None else None,
                                              _ptr(tokens_out), _ptr(logits_out), _stream(stream)),
           "fpd_constrain_argmax_noalloc")


def fpd_verify(mode, batch, block_len, draft, target, layout, rule, pad_id, accept_len, committed, valid_out,
               stream=None):
    _check(lib().fpd_verify(mode, batch, block_len, _ptr(draft), _ptr(target),
                            ctypes.byref(layout) if layout is not None else None, _ptr(rule), int(pad_id),
                            _ptr(accept_len), _ptr(committed), _ptr(valid_out), _stream(stream)), "fpd_verify")


def fpd_verify_prefix(batch, block_len, draft, margin, tau, layout, rule, pad_id, accept_len, committed, valid_out,
                      stream=None):
    _check(lib().fpd_verify_prefix(batch, block_len, _ptr(draft), _ptr(margin), float(tau), ctypes.byref(layout),
                                   _ptr(rule), int(pad_id), _ptr(accept_len), _ptr(committed), _ptr(valid_out),
                                   _stream(stream)), "fpd_verify_prefix")


def grid_format(digit_ids, plus_id, minus_id, pad_id, n_axes=3, width=5, axis_sep=",", point_sep=";") -> GridFormat:
    f = GridFormat()
    for k, t in enumerate(digit_ids):
        f.digit_id[k] = int(t)
    f.plus_id, f.minus_id, f.pad_id, f.n_axes, f.width = int(plus_id), int(minus_id), int(pad_id), n_axes, width
    f.axis_sep, f.point_sep = axis_sep.encode(), point_sep.encode()
    return f


def fpd_grid_to_text(committed, accept, fmt: GridFormat) -> list:
    """Host arrays (numpy int32 [B, L] committed tokens, [B] accepted positions) -> one text per request."""
    import numpy as np
    cm = np.ascontiguousarray(committed, dtype=np.int32)
    acc = np.ascontiguousarray(accept, dtype=np.int32)
    B, L = cm.shape
    cap = B * (L * 4 + 16)
    out = ctypes.create_string_buffer(cap)
    offs = (ctypes.c_size_t * (B + 1))()
    _check(lib().fpd_grid_to_text(B, L, cm.ctypes.data, acc.ctypes.data, ctypes.byref(fmt), out, cap, offs),
           "fpd_grid_to_text")
    return [ctypes.string_at(ctypes.addressof(out) + offs[b]).decode() for b in range(B)]


def fpd_kernel_launches() -> int:
    return int(lib().fpd_kernel_launches())


def fpd_last_error() -> str:
    return lib().fpd_last_error().decode()


def fpd_device_status(stream=None) -> int:
    code = ctypes.c_int32(0)
    st = lib().fpd_device_status(_stream(stream), ctypes.byref(code))
    if st not in (FPD_OK, 6):
        _check(st, "fpd_device_status")
    return int(code.value)


from .drafter import Drafter  # noqa: E402  (convenience wrapper over the calls above)
