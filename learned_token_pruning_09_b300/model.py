"""A synthetic Qwen3-style model run through the library's calls: the
pruned prefill that ends in the first token, and the first decode step over
its caches (TokenGate's three phases, MarkTechPost article, "How does
TokenGate's learned token pruning work?").

Every computation is one of libtokengate's kernels (RMSNorm, projections,
QK-norm, RoPE, token-gated attention, gate, top-K, gather, SwiGLU, decode
attention); this module only allocates tensors and orders the calls.  Layer
layout and readings as in the oracle of the same model: pre-norm RMSNorm,
per-head QK-norm before RoPE, SwiGLU MLP; layers below the gate layer L and
the attention of layer L run on every token, the gate reads layer L's
post-attention residual, the rest runs on the kept rows with the score bias;
the decode step reads full caches in layers 0..L and kept-only caches above.
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np
import torch

from . import tokengate as tg


class SyntheticModel:
    """Device weights (bf16) of a model from ``synth.model_params``."""

    def __init__(self, params: Dict[str, object], device="cuda", theta: float = 1.0e6):
        c = params["config"]
        self.cfg, self.dev, self.theta = c, torch.device(device), theta
        self.hq, self.hkv, self.dh, self.L = c["hq"], c["hkv"], c["head_dim"], c["gate_layer"]

        def bf(a):
            if isinstance(a, torch.Tensor):            # already bf16 on the device
                return a.to(self.dev).contiguous()
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(self.dev).view(torch.bfloat16)

        def f32(a):
            if isinstance(a, torch.Tensor):
                return a.to(device=self.dev, dtype=torch.float32).contiguous()
            return torch.as_tensor(np.asarray(a, np.float32)).to(self.dev)

        self.layers = []
        for lp in params["layers"]:
            self.layers.append({
                "ln1": bf(lp["ln1"]), "ln2": bf(lp["ln2"]), "q_norm": bf(lp["q_norm"]), "k_norm": bf(lp["k_norm"]),
                "w_q": bf(lp["w_q"]), "w_k": bf(lp["w_k"]), "w_v": bf(lp["w_v"]), "w_o": bf(lp["w_o"]),
                "w_gate_up": torch.cat([bf(lp["w_gate"]), bf(lp["w_up"])], dim=0).contiguous(),
                "w_down": bf(lp["w_down"]),
                "gain": f32(lp["gain"]), "tau": float(lp["tau"])})
        g = params["gate"]
        self.gate = {"w1": bf(g["w1"]), "w2": bf(g["w2"]), "b1": f32(g["b1"]), "b2": float(g["b2"])}
        self.final_norm = bf(params["final_norm"])
        self.w_lm = bf(params["w_lm"])
        self.zero_gain = torch.zeros(self.hq, dtype=torch.float32, device=self.dev)

    # ---- blocks ----
    def _attn_block(self, x, li, pos, cu, max_len, s, gain, tau):
        """h = x + attention; returns h and the layer's cache (k' rotated, v)."""
        p, t = self.layers[li], x.shape[0]
        a = tg.tg_rms_norm(x, p["ln1"])
        q = tg.tg_rms_norm(tg.tg_linear_bf16(a, p["w_q"]).view(t, self.hq, self.dh), p["q_norm"])
        k = tg.tg_rms_norm(tg.tg_linear_bf16(a, p["w_k"]).view(t, self.hkv, self.dh), p["k_norm"])
        v = tg.tg_linear_bf16(a, p["w_v"]).view(t, self.hkv, self.dh)
        k_rot = torch.empty_like(k)
        o = tg.tg_gated_attention_fwd(q, k, v, pos, s, gain, tau, self.theta, cu, max_len, k_cache=k_rot)
        h = tg.tg_linear_bf16(o.view(t, self.hq * self.dh), p["w_o"], residual=x)
        return h, (k_rot, v)

    def _mlp_block(self, h, li):
        p = self.layers[li]
        gu = tg.tg_linear_bf16(tg.tg_rms_norm(h, p["ln2"]), p["w_gate_up"])
        return tg.tg_linear_bf16(tg.tg_swiglu(gu), p["w_down"], residual=h)

    def _logits(self, x_last):
        return tg.tg_linear_bf16(tg.tg_rms_norm(x_last, self.final_norm), self.w_lm)

    # ---- the pruned prefill ----
    def prefill(self, x: torch.Tensor, seqlens: Sequence[int], n_doc: Sequence[int], k: Sequence[int]):
        """x [N, d] bf16 input rows of a packed batch.  Returns a dict with
        the logits [B, vocab] (bf16) of each sequence's last row and what the
        decode step needs (caches, kept layout, scores)."""
        dev = self.dev
        seqlens = [int(v) for v in seqlens]
        cu_h = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
        cu = torch.as_tensor(cu_h).to(dev)
        pos = torch.as_tensor(np.concatenate([np.arange(n) for n in seqlens]).astype(np.int32)).to(dev)
        n_rows = int(cu_h[-1])
        zeros_s = torch.zeros(n_rows, dtype=torch.float32, device=dev)
        max_len = max(seqlens)
        caches: List[tuple] = []
        for li in range(self.L):
            h, cache = self._attn_block(x, li, pos, cu, max_len, zeros_s, self.zero_gain, 1.0)
            caches.append(cache)
            x = self._mlp_block(h, li)
        h, cache = self._attn_block(x, self.L, pos, cu, max_len, zeros_s, self.zero_gain, 1.0)
        caches.append(cache)
        nd = torch.as_tensor(np.asarray(n_doc, np.int32)).to(dev)
        ws = tg.tg_topk_workspace(len(seqlens), dev)
        s = tg.tg_gate_score(h, cu, nd, self.gate["w1"], self.gate["b1"], self.gate["w2"], self.gate["b2"],
                             topk_ws=ws)
        kept_len = tg.kept_lengths(seqlens, n_doc, k)
        n_kept = int(sum(kept_len))
        kept, cu_kept = tg.tg_topk_select(s, cu, nd, torch.as_tensor(np.asarray(k, np.int32)).to(dev), max(n_doc),
                                          n_kept, workspace=ws)
        hk, pos_k, s_k = tg.tg_gather_kept(h, s, cu, kept, cu_kept, n_kept)
        xk = self._mlp_block(hk, self.L)
        max_kept = max(kept_len)
        for li in range(self.L + 1, len(self.layers)):
            p = self.layers[li]
            h, cache = self._attn_block(xk, li, pos_k, cu_kept, max_kept, s_k, p["gain"], p["tau"])
            caches.append(cache)
            xk = self._mlp_block(h, li)
        # each sequence's last kept row (its last question token) gives the first token's logits
        last = torch.as_tensor((np.cumsum(kept_len) - 1).astype(np.int32)).to(dev)
        cu_rows = torch.as_tensor(np.arange(len(seqlens) + 1, dtype=np.int32)).to(dev)
        cu_kept_full = torch.as_tensor(np.concatenate([[0], np.cumsum(kept_len)]).astype(np.int32)).to(dev)
        x_last, _, _ = tg.tg_gather_kept(xk, None, cu_kept_full, last, cu_rows, len(seqlens), want=("x",))
        return {"logits": self._logits(x_last), "caches": caches, "cu": cu, "seqlens": seqlens, "cu_kept": cu_kept,
                "kept_len": kept_len, "s_kept": s_k, "kept": kept, "pruned": True}

    # ---- the full (unpruned) prefill, the baseline TokenGate is measured against ----
    def prefill_full(self, x: torch.Tensor, seqlens: Sequence[int]):
        """Every layer on every row with plain causal attention (no gate, no
        score bias): the full prefill.  Returns the logits [B, vocab] of each
        sequence's last row and the full-length caches of every layer."""
        dev = self.dev
        seqlens = [int(v) for v in seqlens]
        cu_h = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
        cu = torch.as_tensor(cu_h).to(dev)
        pos = torch.as_tensor(np.concatenate([np.arange(n) for n in seqlens]).astype(np.int32)).to(dev)
        zeros_s = torch.zeros(int(cu_h[-1]), dtype=torch.float32, device=dev)
        caches: List[tuple] = []
        for li in range(len(self.layers)):
            h, cache = self._attn_block(x, li, pos, cu, max(seqlens), zeros_s, self.zero_gain, 1.0)
            caches.append(cache)
            x = self._mlp_block(h, li)
        last = torch.as_tensor((cu_h[1:] - 1).astype(np.int32)).to(dev)
        cu_rows = torch.as_tensor(np.arange(len(seqlens) + 1, dtype=np.int32)).to(dev)
        x_last, _, _ = tg.tg_gather_kept(x, None, cu, last, cu_rows, len(seqlens), want=("x",))
        return {"logits": self._logits(x_last), "caches": caches, "cu": cu, "seqlens": seqlens, "pruned": False}

    # ---- the first decode step ----
    def decode(self, x_new: torch.Tensor, state: Dict[str, object]):
        """x_new [B, d] bf16: the input row of each sequence's generated token
        (at position N_b), over the caches of ``prefill`` (kept-only above the
        gate layer) or ``prefill_full`` (full length everywhere).  Returns the
        next logits [B, vocab] (bf16)."""
        dev, b = self.dev, x_new.shape[0]
        cu_b = torch.as_tensor(np.arange(b + 1, dtype=np.int32)).to(dev)
        pos_new = torch.as_tensor(np.asarray(state["seqlens"], np.int32)).to(dev)
        x = x_new
        for li, p in enumerate(self.layers):
            a = tg.tg_rms_norm(x, p["ln1"])
            q = tg.tg_rms_norm(tg.tg_linear_bf16(a, p["w_q"]).view(b, self.hq, self.dh), p["q_norm"])
            k = tg.tg_rms_norm(tg.tg_linear_bf16(a, p["w_k"]).view(b, self.hkv, self.dh), p["k_norm"])
            v = tg.tg_linear_bf16(a, p["w_v"]).view(b, self.hkv, self.dh)
            q_rot, k_rot = tg.tg_rope_qk(q, k, pos_new, self.theta, cu_b)
            k_c, v_c = state["caches"][li]
            if state["pruned"] and li > self.L:
                o = tg.tg_decode_attention(q_rot, k_rot, v, k_c, v_c, state["cu_kept"], max(state["kept_len"]),
                                           s_cache=state["s_kept"], gain=p["gain"], tau=p["tau"])
            else:
                o = tg.tg_decode_attention(q_rot, k_rot, v, k_c, v_c, state["cu"], max(state["seqlens"]))
            h = tg.tg_linear_bf16(o.view(b, self.hq * self.dh), p["w_o"], residual=x)
            x = self._mlp_block(h, li)
        return self._logits(x)
