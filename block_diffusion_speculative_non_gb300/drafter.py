"""Convenience wrapper: device copies of the weights, the model handle, the KV store and the workspace.

Marshalling only — each method is one C-ABI call.  Weights arrive as bf16 bit patterns (numpy uint16) or
torch bf16 tensors and are copied to the device once.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (FPD_VERIFY_SCHEMA, FPD_VERIFY_TEXT, MAX_LAYERS, ModelDesc, Weights, fpd_constrain_argmax,
               fpd_draft_block, fpd_kv_store_bytes, fpd_model_create, fpd_model_destroy, fpd_model_enable_fp8,
               fpd_prepare_context,
               fpd_prepare_context_rows, fpd_sd_advance, fpd_verify, fpd_verify_prefix, fpd_workspace_bytes,
               make_layout)

_LAYER_KEYS = ("attn_norm", "wqkv", "q_norm", "k_norm", "wo", "mlp_norm", "w_gate_up", "w_down")


def to_device_bf16(a, device) -> torch.Tensor:
    if isinstance(a, torch.Tensor):
        return a.to(device=device, dtype=torch.bfloat16).contiguous()
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)


class Drafter:
    """One drafter model on one GPU, sized for up to `max_batch` requests of `t_cap` context positions and
    blocks of up to `max_block_len` positions.  fp8=True adds the 8-bit copies of the streamed matrices
    (fpd_model_enable_fp8): calls of at most 16 positions then run on them."""

    def __init__(self, shape, weights, max_batch: int, max_block_len: int, t_cap: int, device="cuda", fp8=False):
        self.shape = shape
        self.device = torch.device(device)
        self.max_batch, self.max_block_len, self.t_cap = max_batch, max_block_len, t_cap
        self.w = {k: to_device_bf16(weights[k], self.device) for k in ("embed", "w_fc", "hidden_norm", "final_norm",
                                                                       "lm_head")}
        self.layers = [{k: to_device_bf16(lw[k], self.device) for k in _LAYER_KEYS} for lw in weights["layers"]]
        desc = ModelDesc(shape.n_layers, shape.d_model, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.d_ff,
                         shape.vocab, shape.n_feat, t_cap + max_block_len, shape.rms_eps, shape.rope_theta)
        W = Weights()
        for k, t in self.w.items():
            setattr(W, k, t.data_ptr())
        for name in _LAYER_KEYS:
            arr = (getattr(W, name))
            for l in range(shape.n_layers):
                arr[l] = self.layers[l][name].data_ptr()
        self.handle = fpd_model_create(desc, W)
        if fp8:
            fpd_model_enable_fp8(self.handle)
        self.kv_bytes = fpd_kv_store_bytes(self.handle, max_batch, t_cap)
        self.ws_bytes = fpd_workspace_bytes(self.handle, max_batch, max_block_len, t_cap)
        self.kv_store = torch.zeros(self.kv_bytes // 2, dtype=torch.bfloat16, device=self.device)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)

    def close(self):
        if getattr(self, "handle", None):
            fpd_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kv_view(self, batch=None):
        s = self.shape
        B = self.max_batch if batch is None else batch
        return self.kv_store[: s.n_layers * B * 2 * s.n_kv_heads * self.t_cap * s.head_dim].view(
            s.n_layers, B, 2, s.n_kv_heads, self.t_cap, s.head_dim)

    # ---- calls ----------------------------------------------------------------------------------------------
    def prepare_context(self, batch, row_off, feats, pos_start=None, stream=None):
        total = int(row_off[-1].item()) if isinstance(row_off, torch.Tensor) else int(row_off[-1])
        row_off_d = torch.as_tensor(np.asarray(row_off, dtype=np.int32) if not isinstance(row_off, torch.Tensor)
                                    else row_off, device=self.device, dtype=torch.int32)
        ps = None if pos_start is None else torch.as_tensor(pos_start, device=self.device, dtype=torch.int32)
        fd = [to_device_bf16(f, self.device) for f in feats]
        fpd_prepare_context(self.handle, batch, total, row_off_d, ps, fd, self.kv_store, self.t_cap, self.workspace,
                            self.ws_bytes, stream)
        return fd, row_off_d, ps

    def draft_block(self, batch, block_len, ctx_len, anchor, mask_id, hidden_out=None, layer_hidden=None,
                    stream=None):
        s = self.shape
        if hidden_out is None:
            hidden_out = torch.empty(batch * block_len, s.d_model, dtype=torch.bfloat16, device=self.device)
        fpd_draft_block(self.handle, batch, block_len, self.kv_store, self.t_cap, ctx_len, anchor, mask_id, hidden_out,
                        layer_hidden, self.workspace, self.ws_bytes, stream)
        return hidden_out

    def constrain_argmax(self, batch, block_len, hidden, layout=None, tokens_out=None, logits_out=None, stream=None,
                         margin_out=None):
        if tokens_out is None:
            tokens_out = torch.empty(batch, block_len - 1, dtype=torch.int32, device=self.device)
        fpd_constrain_argmax(self.handle, batch, block_len, hidden, layout, tokens_out, logits_out, self.workspace,
                             self.ws_bytes, stream, margin_out=margin_out)
        return tokens_out

    def prepare_rows(self, batch, total_rows, row_off_d, row_cnt_d, pos_start_d, feats_d, stream=None):
        """fpd_prepare_context_rows on device arrays (appends whose row counts live on the device)."""
        fpd_prepare_context_rows(self.handle, batch, total_rows, row_off_d, row_cnt_d, pos_start_d, feats_d,
                                 self.kv_store, self.t_cap, self.workspace, self.ws_bytes, stream)

    def verify_prefix(self, batch, block_len, draft, margin, tau, layout, rule, pad_id, stream=None):
        """Primitive acceptance keeping the prefix before the first failing or uncertain position."""
        dev = self.device
        accept = torch.empty(batch, dtype=torch.int32, device=dev)
        committed = torch.empty(batch, block_len, dtype=torch.int32, device=dev)
        valid = torch.empty(batch, dtype=torch.int32, device=dev)
        fpd_verify_prefix(batch, block_len, draft, margin, tau, layout, rule, pad_id, accept, committed, valid, stream)
        return accept, committed, valid

    def spec_state(self, batch, block_len, ctx_len, anchor):
        """Device buffers of a text speculative loop (see spec_step), starting from ctx_len / anchor."""
        return SpecState(self, batch, block_len, ctx_len, anchor)

    def spec_step(self, st, feats_d, make_target, mask_id, stream=None, logits_out=None):
        """One text speculative step on the device, with no host synchronisation (capturable in a CUDA graph):
        draft block -> unconstrained argmax -> make_target(st.tokens, st.target) (the target model's greedy row for
        the drafted block; the caller supplies it) -> text verification -> fpd_sd_advance -> append of the target's
        features at the accepted positions.  feats_d: n_feat device tensors [batch * block_len, d]; row
        b * block_len + j holds request b's feature at block position j (anchor j = 0)."""
        B, L = st.batch, st.block_len
        self.draft_block(B, L, st.ctx_len, st.anchor, mask_id, hidden_out=st.hidden, stream=stream)
        self.constrain_argmax(B, L, st.hidden, tokens_out=st.tokens, logits_out=logits_out, stream=stream)
        make_target(st.tokens, st.target)
        fpd_verify(0, B, L, st.tokens, st.target, None, None, -1, st.accept, st.committed, st.valid, stream)
        st.after_verify(stream)
        fpd_sd_advance(B, L, self.t_cap, st.accept, st.committed, st.ctx_len, st.pos_start, st.anchor, stream)
        self.prepare_rows(B, B * L, st.row_off, st.accept, st.pos_start, feats_d, stream)

    @staticmethod
    def layout(layout_np: dict, batch: int, block_len: int, device="cuda"):
        """Device copy of a layout dict (class tables stay on the host)."""
        pc = np.asarray(layout_np["pos_class"], dtype=np.int16)
        if pc.ndim == 1:
            pc = np.broadcast_to(pc, (batch, block_len))
        pc_d = torch.from_numpy(np.array(pc, dtype=np.int16, order="C", copy=True)).to(device)
        lay = make_layout(layout_np["class_off"], layout_np["class_ranges"], pc_d, pairs=layout_np.get("pairs"),
                          off_id=layout_np.get("off_id", 0))
        rule = layout_np.get("rule")
        rule_d = None
        if rule is not None:
            r = np.asarray(rule, dtype=np.int8)
            if r.ndim == 1:
                r = np.broadcast_to(r, (batch, block_len))
            rule_d = torch.from_numpy(np.array(r, dtype=np.int8, order="C", copy=True)).to(device)
        return lay, rule_d

    def verify_text(self, batch, block_len, draft, target, accept=None, committed=None, valid=None, stream=None):
        dev = self.device
        accept = torch.empty(batch, dtype=torch.int32, device=dev) if accept is None else accept
        committed = torch.empty(batch, block_len, dtype=torch.int32, device=dev) if committed is None else committed
        valid = torch.empty(batch, dtype=torch.int32, device=dev) if valid is None else valid
        fpd_verify(FPD_VERIFY_TEXT, batch, block_len, draft, target, None, None, -1, accept, committed, valid, stream)
        return accept, committed, valid

    def verify_schema(self, batch, block_len, draft, layout, rule, pad_id, accept=None, committed=None, valid=None,
                      stream=None):
        dev = self.device
        accept = torch.empty(batch, dtype=torch.int32, device=dev) if accept is None else accept
        committed = torch.empty(batch, block_len, dtype=torch.int32, device=dev) if committed is None else committed
        valid = torch.empty(batch, dtype=torch.int32, device=dev) if valid is None else valid
        fpd_verify(FPD_VERIFY_SCHEMA, batch, block_len, draft, None, layout, rule, pad_id, accept, committed, valid,
                   stream)
        return accept, committed, valid


class SpecState:
    """Device state of a text speculative loop: context lengths, anchors, the step's outputs, and the fixed
    row offsets (block_len rows per request) of the feature buffer an append reads."""

    def __init__(self, dr, batch, block_len, ctx_len, anchor):
        dev = dr.device
        i32 = dict(dtype=torch.int32, device=dev)
        self.batch, self.block_len = batch, block_len
        self.ctx_len = torch.as_tensor(np.asarray(ctx_len, np.int32), **i32).clone()
        self.anchor = torch.as_tensor(np.asarray(anchor, np.int32), **i32).clone()
        self.pos_start = torch.zeros(batch, **i32)
        self.accept = torch.zeros(batch, **i32)
        self.committed = torch.zeros(batch, block_len, **i32)
        self.valid = torch.zeros(batch, **i32)
        self.tokens = torch.zeros(batch, block_len - 1, **i32)
        self.target = torch.zeros(batch, block_len, **i32)
        self.hidden = torch.empty(batch * block_len, dr.shape.d_model, dtype=torch.bfloat16, device=dev)
        self.row_off = torch.arange(0, (batch + 1) * block_len, block_len, **i32)
        self.hooks = []

    def after_verify(self, stream=None):
        for h in self.hooks:   # callers record per-step results here (e.g. copies into a history buffer)
            h(self)
