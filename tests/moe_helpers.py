"""Shared test helpers: build one MoE layer for both the CUDA path and the
oracle from the same seeded inputs, and the forward tolerance check.

Forward tolerance (derived; the same bound everywhere):
    |gpu_i - ref_i| <= 1e-2 * rms(ref) + |ref_i| * 2^-8
The first term is the 1e-2 RMS-normalised bound; the second is the largest
possible error of rounding a correct value to the bf16 output format (half
an ulp, at most 2^-8 relative).  Without it, output rounding alone breaks a
pure 1e-2 bound at the output's outliers once a few hundred thousand values
are compared.
"""

import numpy as np
import torch

import oracle
from weight_quantized_moe_gb300 import synth

FWD_TOL = 1e-2


def forward_error(got, ref):
    """max_i (|got_i - ref_i| - |ref_i| 2^-8)_+ / rms(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    if rms == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    excess = np.maximum(np.abs(got - ref) - np.abs(ref) * 2.0 ** -8, 0.0)
    return float(excess.max() / rms)


def plain_error(got, ref):
    """max_i |got_i - ref_i| / rms(ref), without the output-rounding term."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    if rms == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / rms) if got.size else 0.0


def check_forward(got, ref, tol=FWD_TOL, what=""):
    """Assert the forward tolerance; the message gives both the bound's
    figure and the plain max |err| / rms beside it."""
    err = forward_error(got, ref)
    plain = plain_error(got, ref)
    assert err <= tol, (f"{what} forward error {err:.3e} > {tol:.0e} "
                        f"(plain max|err|/rms {plain:.3e})")
    return err, plain


def route_tolerance(E):
    """Relative bound on |w_gpu - w_ref| / w_ref for float32 softmax weights:
    E-term float32 sum plus exp and the final division, each a few units of
    float32 roundoff (2^-24)."""
    return (E + 8) * 2.0 ** -24 * 4


class Layer:
    """One synthetic layer on the device, with lazy oracle-side weights."""

    def __init__(self, wl, seed=0, device="cuda", gen_device=None):
        self.wl = wl
        self.E, self.k, self.H, self.I = wl.E, wl.k, wl.H, wl.I
        self.bits, self.gs, self.has_zp = wl.bits, wl.group_size, wl.has_zp
        self.seed = seed
        self.device = device
        self.gen_device = gen_device or device
        import weight_quantized_moe_gb300 as mq
        E, H, I = self.E, self.H, self.I
        w13 = synth.expert_weights(E, 2 * I, H, seed, "w13", device=self.gen_device).to(device)
        w2 = synth.expert_weights(E, H, I, seed, "w2", device=self.gen_device).to(device)
        self._bf16 = (w13, w2)
        if self.bits == 8:
            self.q13, self.s13 = mq.moe_quantize_int8_per_channel(w13)
            self.q2, self.s2 = mq.moe_quantize_int8_per_channel(w2)
            self.z13 = self.z2 = None
        else:
            self.q13, self.s13, self.z13 = mq.moe_quantize_uint4_group(w13, self.gs)
            self.q2, self.s2, self.z2 = mq.moe_quantize_uint4_group(w2, self.gs)
        self._oracle = {}

    def bf16_expert(self, e, which):
        t = self._bf16[0] if which == "w13" else self._bf16[1]
        return t[e].float().cpu().numpy()

    def free_bf16(self):
        self._bf16 = (None, None)

    def forward(self, x, topk_w, topk_ids, **kw):
        import weight_quantized_moe_gb300 as mq
        return mq.moe_quant_forward(x, self.q13, self.q2, self.s13, self.s2, topk_w, topk_ids,
                                    bits=self.bits, group_size=self.gs, has_zp=self.has_zp,
                                    z13=self.z13, z2=self.z2, **kw)

    # ---- oracle side: the oracle quantises the same bf16 weights itself ----
    def oracle_experts(self, experts=None):
        """Oracle Int8Experts/Uint4Experts holding the given experts (others
        zero).  Quantised by the oracle from the bf16 weights."""
        E, H, I = self.E, self.H, self.I
        experts = range(E) if experts is None else sorted(set(int(e) for e in experts))
        if self.bits == 8:
            ex = oracle.Int8Experts(np.zeros((E, 2 * I, H), np.int8), np.zeros((E, 2 * I), np.float32),
                                    np.zeros((E, H, I), np.int8), np.zeros((E, H), np.float32))
            for e in experts:
                ex.w13[e], ex.s13[e] = self._oracle_int8(e, "w13")
                ex.w2[e], ex.s2[e] = self._oracle_int8(e, "w2")
            return ex
        gs = self.gs
        ex = oracle.Uint4Experts(
            np.zeros((E, 2 * I, H // 2), np.uint8), np.zeros((E, 2 * I, H // gs), np.float16),
            np.zeros((E, I, H // gs), np.uint8), np.zeros((E, H, I // 2), np.uint8),
            np.zeros((E, H, I // gs), np.float16), np.zeros((E, H // 2, I // gs), np.uint8),
            gs, self.has_zp)
        for e in experts:
            ex.qw13[e], ex.sc13[e], ex.qz13[e] = self._oracle_uint4(e, "w13")
            ex.qw2[e], ex.sc2[e], ex.qz2[e] = self._oracle_uint4(e, "w2")
        return ex

    def _oracle_int8(self, e, which):
        key = ("i8", e, which)
        if key not in self._oracle:
            self._oracle[key] = oracle.quantize_int8_per_channel(self.bf16_expert(e, which))
        return self._oracle[key]

    def _oracle_uint4(self, e, which):
        key = ("u4", e, which)
        if key not in self._oracle:
            q, s, z = oracle.quantize_uint4_group(self.bf16_expert(e, which), self.gs)
            self._oracle[key] = (oracle.pack_uint4_along_k(q), s, oracle.pack_uint4_along_n(z))
        return self._oracle[key]


def inputs(wl, T, seed=0, device="cuda"):
    x = synth.hidden_states(T, wl.H, seed, device=device)
    lg = synth.router_logits(T, wl.E, seed, bias=wl.bias, device=device)
    return x, lg
