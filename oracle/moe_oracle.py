"""Plain, slow, obviously-correct numpy restatement of the quantised MoE path.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing in the CUDA
library imports, links or calls this module.

Sources (vLLM API documentation pages):

* P-int8  = "vllm.model_executor.layers.quantization.experts_int8"
    - ``quantize_in_place_and_get_scales``: the per-output-row int8 quantiser.
    - ``ExpertsInt8MoEMethod.create_weights``: w13 int8 [E, 2I, H],
      w2 int8 [E, H, I], w13_scale fp32 [E, 2I], w2_scale fp32 [E, H].
    - ``ExpertsInt8MoEMethod.quantizing_weight_loader``: gate (w1) rows fill
      w13[:, 0:I], up (w3) rows fill w13[:, I:2I]; w2 rows are quantised per
      row of H.
    - ``ExpertsInt8MoEMethod.apply``: select_experts (softmax scoring, top_k,
      renormalize) followed by fused_experts with activation "silu" and the
      per-channel scales.
* P-wna16 = "vllm.model_executor.layers.quantization.moe_wna16"
    - ``MoeWNA16Method.create_weights``: packed uint8 qweight [E, N, K/2],
      scales [E, N, K/gs], qzeros uint8 [E, N/2, K/gs] (packed along N).
    - ``get_weight_loader.convert_awq_tensor`` step 5: two 4-bit values per
      byte, the even index in the low nibble.
    - ``get_weight_loader.convert_gptq_int4_qzeros``: GPTQ stores z-1, the
      loader adds 1, so the stored zero is the true zero point.
    - ``MoeWNA16Method`` with ``num_bits == 8``: ``group_size == -1`` (one
      group per output row), qweight uint8 [E, N, K] (``bit8_pack_factor``
      1), scales [E, N, 1] in the parameter dtype, optional qzeros uint8
      [E, N, 1] (for 8 bits the loader also adds 1 to GPTQ zeros).
* P-ct = "vllm.model_executor.layers.fused_moe.oracle.int8" (compressed-
  tensors int8 config): strategy "channel", or "tensor" when the weight
  scale has fewer elements than experts x output rows -- one scale per
  expert.
* P-int8 ``ExpertsInt8MoEMethod.apply`` passes ``apply_router_weight_on_input``
  through to ``fused_experts``; the supported activation dtypes are bf16 and
  fp16.
* P-int8 ``ExpertsInt8MoEMethod.apply`` and P-wna16
  ``MoeWNA16Method.apply_monolithic`` name the further router arguments
  (``scoring_func``, ``num_expert_group`` / ``topk_group``,
  ``e_score_correction_bias``, ``routed_scaling_factor``) without their
  arithmetic; ``topk_route_ex`` states the reading taken.

Readings taken where the pages are silent are marked "Reading:" in place.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_F32 = np.float32
_INT8_VMAX = 127  # torch.iinfo(torch.int8).max, used for both scale and clamp


# --------------------------------------------------------------------------
# W8A16: int8 per-output-channel quantiser (P-int8,
# quantize_in_place_and_get_scales)
# --------------------------------------------------------------------------
def quantize_int8_per_channel(w):
    """Quantise each row of ``w`` [R, C] to int8 with one fp32 scale per row.

    Steps, in the page's order: scale = max_c |w[r, c]| / 127; w / scale;
    round half to even (torch ``round_``); clamp to [-127, 127].

    Reading (dtype): every step runs in float32 (the page runs them in the
    loaded tensor's dtype, which it does not fix; the scale parameter it
    fills is float32).  The division is a true IEEE float32 division, not a
    multiply by a reciprocal.
    Reading (all-zero row): the page would divide 0 by 0; here such a row
    gets scale 0 and codes 0, so it dequantises to exact zeros.

    Returns (q int8 [R, C], scale float32 [R]).
    """
    w = np.asarray(w, dtype=_F32)
    if w.ndim != 2:
        raise ValueError("w must be 2-D [rows, cols]")
    amax = np.max(np.abs(w), axis=1) if w.shape[1] else np.zeros(w.shape[0], _F32)
    scale = (amax / _F32(_INT8_VMAX)).astype(_F32)
    q = np.zeros(w.shape, dtype=np.int8)
    live = scale > 0
    if np.any(live):
        ratio = (w[live] / scale[live, None]).astype(_F32)
        q[live] = np.clip(np.rint(ratio), -_INT8_VMAX, _INT8_VMAX).astype(np.int8)
    return q, scale


def dequantize_int8_per_channel(q, scale):
    """w_hat[r, c] = q[r, c] * scale[r], in float64."""
    return np.asarray(q, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[..., None]


# --------------------------------------------------------------------------
# W4A16: uint4 group quantisation (input helper) and the P-wna16 storage
# --------------------------------------------------------------------------
def quantize_uint4_group(w, group_size):
    """Asymmetric uint4 quantisation of ``w`` [R, C] in groups along C.

    The pages only consume already-quantised GPTQ/AWQ tensors, so this
    quantiser exists to make test and benchmark inputs.  Reading: the usual
    min-max scheme with the range widened to include zero, per group g:

        lo = min(0, min w_g), hi = max(0, max w_g)
        s  = fp16((hi - lo) / 15)            (float32 division, then fp16 RNE)
        z  = clamp(rint(-lo / s), 0, 15)
        q  = clamp(rint(w / s) + z, 0, 15)
        dequant = (q - z) * s

    A group whose fp16 scale is 0 gets z = 0 and q = 0 (dequantises to 0).
    Returns (q uint8 [R, C] values 0..15, s float16 [R, C/gs], z uint8 [R, C/gs]).
    """
    w = np.asarray(w, dtype=_F32)
    R, C = w.shape
    if group_size <= 0 or C % group_size:
        raise ValueError("group_size must divide the row length")
    G = C // group_size
    wg = w.reshape(R, G, group_size)
    lo = np.minimum(wg.min(axis=2), _F32(0))
    hi = np.maximum(wg.max(axis=2), _F32(0))
    s16 = ((hi - lo).astype(_F32) / _F32(15)).astype(_F32).astype(np.float16)
    s = s16.astype(_F32)
    z = np.zeros((R, G), dtype=np.uint8)
    q = np.zeros((R, G, group_size), dtype=np.uint8)
    live = s > 0
    if np.any(live):
        zl = np.clip(np.rint((-lo[live]) / s[live]), 0, 15)
        z[live] = zl.astype(np.uint8)
        ql = np.rint((wg[live] / s[live][:, None]).astype(_F32)) + zl[:, None]
        q[live] = np.clip(ql, 0, 15).astype(np.uint8)
    return q.reshape(R, C), s16, z


def pack_uint4_along_k(q):
    """[.., K] values 0..15 -> uint8 [.., K/2]; byte j = q[2j] | q[2j+1] << 4.

    Low nibble holds the even index, as the AWQ repack of P-wna16 lands on
    (odd-index value times 16 plus even-index value).
    """
    q = np.asarray(q, dtype=np.uint8)
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def unpack_uint4_along_k(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def pack_uint4_along_n(z):
    """Zero points [.., N, G] -> uint8 [.., N/2, G]; row 2i in the low nibble.

    P-wna16 packs qzeros along the output dimension (shape
    [E, 2I / pack_factor, H / gs]) with the even row in the low nibble.
    """
    z = np.asarray(z, dtype=np.uint8)
    return (z[..., 0::2, :] | (z[..., 1::2, :] << 4)).astype(np.uint8)


def unpack_uint4_along_n(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-2] + (p.shape[-2] * 2, p.shape[-1]), dtype=np.uint8)
    out[..., 0::2, :] = p & 0xF
    out[..., 1::2, :] = p >> 4
    return out


def dequantize_uint4_group(qpacked, scales, zpacked, group_size, has_zp=True):
    """(q - z) * s per group along K, in float64, for one expert's matrix.

    qpacked uint8 [N, K/2], scales fp16 [N, K/gs], zpacked uint8 [N/2, K/gs].
    Reading (has_zp false, symmetric GPTQ): the implicit zero is 8, the
    middle of the 4-bit range.
    """
    q = unpack_uint4_along_k(qpacked).astype(np.float64)
    N, K = q.shape
    G = K // group_size
    if has_zp:
        z = unpack_uint4_along_n(zpacked).astype(np.float64)
    else:
        z = np.full((N, G), 8.0)
    s = np.asarray(scales).astype(np.float64)
    qg = q.reshape(N, G, group_size)
    return ((qg - z[:, :, None]) * s[:, :, None]).reshape(N, K)


# --------------------------------------------------------------------------
# Router: softmax -> top-k -> renormalise (P-int8, ExpertsInt8MoEMethod.apply
# passes scoring_func="softmax", top_k, renormalize to select_experts)
# --------------------------------------------------------------------------
def topk_route(logits, k, renormalize):
    """Return (topk_weights float64 [T, k], topk_ids int32 [T, k]).

    Reading (select_experts body is not on the pages): p = softmax over the
    E logits of a token; the k experts with the largest p are chosen.  Since
    softmax is monotone the choice is made on the float32 logits themselves,
    ties going to the lower expert index; slots j = 0..k-1 run from the
    largest to the smallest.  Weight j is p[id_j], divided by the sum over
    the k chosen experts when ``renormalize`` is set.
    """
    logits = np.asarray(logits, dtype=_F32)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    idx = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((idx, -logits.astype(np.float64)), axis=-1)
    ids = order[:, :k].astype(np.int32)
    l64 = logits.astype(np.float64)
    m = l64.max(axis=1, keepdims=True)
    ex = np.exp(l64 - m)
    p = ex / ex.sum(axis=1, keepdims=True)
    w = np.take_along_axis(p, ids, axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return w, ids


def _scores_f32(logits, scoring_func):
    """Float32 scores of every expert, in the order the router kernel forms
    them: softmax as exp(l - max) / sum, sigmoid as 1 / (1 + exp(-l))."""
    l32 = np.asarray(logits, dtype=_F32)
    if scoring_func == "softmax":
        ex = np.exp(l32 - l32.max(axis=1, keepdims=True))
        return ex / ex.sum(axis=1, keepdims=True, dtype=_F32)
    return _F32(1) / (_F32(1) + np.exp(-l32))


def topk_route_ex(logits, k, renormalize, scoring_func="softmax", num_expert_group=0,
                  topk_group=0, e_score_correction_bias=None, routed_scaling_factor=1.0):
    """Router with the extra select_experts arguments: returns (topk_weights
    float64 [T, k], topk_ids int32 [T, k]).

    ``ExpertsInt8MoEMethod.apply`` and ``MoeWNA16Method.apply_monolithic``
    hand ``scoring_func``, ``use_grouped_topk`` / ``num_expert_group`` /
    ``topk_group``, ``e_score_correction_bias`` and
    ``routed_scaling_factor`` to the router; the pages name them and give no
    arithmetic.  Reading, step by step:

    1. Score s_e of each expert: softmax over the token's E logits, or
       sigmoid(logit_e) when ``scoring_func == "sigmoid"``.
    2. Selection key c_e: the logit itself when there is no correction bias
       (either score is increasing in the logit, so this is the order of
       s_e); with a bias b, c_e = s_e + b_e, formed in float32, the
       precision the router kernel decides in.
    3. Grouping (``num_expert_group`` G > 1): experts [gE/G, (g+1)E/G) form
       group g, whose score is the largest key in it.  The ``topk_group``
       groups with the largest scores (ties: lower group) stay; every expert
       of the other groups is out.
    4. Of the experts left, the k with the largest keys (ties: lower index)
       fill slots j = 0..k-1 from the largest key down.
    5. Weight j = s_{id_j}: the bias steers the choice only.  With
       ``renormalize`` it is divided by the sum over the k chosen; then it is
       multiplied by ``routed_scaling_factor``.

    With the defaults this is ``topk_route``.
    """
    logits = np.asarray(logits, dtype=_F32)
    T, E = logits.shape
    if scoring_func not in ("softmax", "sigmoid"):
        raise ValueError("scoring_func must be 'softmax' or 'sigmoid'")
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    G = num_expert_group if num_expert_group and num_expert_group > 1 else 1
    if G > 1:
        if E % G:
            raise ValueError("num_expert_group must divide E")
        if not 1 <= topk_group <= G:
            raise ValueError("need 1 <= topk_group <= num_expert_group")
        if k > topk_group * (E // G):
            raise ValueError("k exceeds the experts of the kept groups")

    # step 1, float64 (the weights); step 2, the keys
    l64 = logits.astype(np.float64)
    if scoring_func == "softmax":
        ex = np.exp(l64 - l64.max(axis=1, keepdims=True))
        score = ex / ex.sum(axis=1, keepdims=True)
    else:
        score = 1.0 / (1.0 + np.exp(-l64))
    if e_score_correction_bias is None:
        key = logits.copy()
    else:
        b32 = np.asarray(e_score_correction_bias, dtype=_F32).reshape(E)
        key = _scores_f32(logits, scoring_func) + b32[None, :]
    key = np.where(np.isnan(key), -np.inf, key).astype(_F32)

    ids = np.zeros((T, k), np.int32)
    for t in range(T):
        allowed = np.ones(E, bool)
        if G > 1:
            gsz = E // G
            gscore = key[t].reshape(G, gsz).max(axis=1)
            # step 3: groups by score, ties to the lower group
            gorder = np.lexsort((np.arange(G), -gscore.astype(np.float64)))
            keep = np.zeros(G, bool)
            keep[gorder[:topk_group]] = True
            allowed = np.repeat(keep, gsz)
        cand = np.nonzero(allowed)[0]
        # step 4: experts by key, ties to the lower index
        order = cand[np.lexsort((cand, -key[t, cand].astype(np.float64)))]
        ids[t] = order[:k]

    w = np.take_along_axis(score, ids, axis=1)   # step 5
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return w * float(routed_scaling_factor), ids


# --------------------------------------------------------------------------
# Block alignment (implied by fused_experts' grouped GEMM; not on the pages)
# --------------------------------------------------------------------------
def align_capacity(T, k, E, block_m):
    """Worst-case padded length: every non-empty expert wastes < block_m rows."""
    S = T * k
    cap = S + min(E, S) * (block_m - 1)
    return -(-cap // block_m) * block_m


@dataclass
class AlignResult:
    sorted_slot_ids: np.ndarray  # int32 [num_padded]; padding = S
    block_expert: np.ndarray     # int32 [num_padded / block_m]
    expert_offsets: np.ndarray   # int32 [E + 1]; [E] == num_padded
    num_padded: int
    invalid_slots: int           # slots whose id lies outside [0, E)


def align_block(topk_ids, E, block_m):
    """Stable counting sort of the token-slots by expert, padded per expert.

    Reading: slot s = t * k + j.  Expert segments follow in expert order; a
    segment holds the slots routed to that expert in increasing s, then the
    sentinel S (= T * k) up to the next multiple of block_m.  An expert with
    no slots gets no block.  A slot whose id is outside [0, E) is placed
    nowhere and counted in ``invalid_slots``.
    """
    ids = np.asarray(topk_ids).reshape(-1).astype(np.int64)
    S = ids.size
    valid = (ids >= 0) & (ids < E)
    counts = np.bincount(ids[valid], minlength=E)[:E]
    padded = -(-counts // block_m) * block_m
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    num_padded = int(offsets[E])
    sorted_ids = np.full(num_padded, S, dtype=np.int32)
    block_expert = np.empty(num_padded // block_m, dtype=np.int32)
    for e in range(E):
        slots = np.nonzero(ids == e)[0]
        sorted_ids[offsets[e]:offsets[e] + slots.size] = slots
        block_expert[offsets[e] // block_m:offsets[e + 1] // block_m] = e
    return AlignResult(sorted_ids, block_expert, offsets.astype(np.int32),
                       num_padded, int(S - valid.sum()))


# --------------------------------------------------------------------------
# Expert weights and the forward (P-int8 apply -> fused_experts)
# --------------------------------------------------------------------------
def round_to_bf16(a):
    """Round to the nearest bfloat16 (ties to even), returned as float64.

    A bfloat16 is the top 16 bits of a float32; the value is first rounded
    to float32, then the low 16 bits are rounded away.  (NaN/inf are not
    expected here.)
    """
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    bits = ((bits + 0x7FFF + lsb) >> 16) << 16
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def silu(u):
    """silu(u) = u / (1 + exp(-u)), the "silu" activation of apply()."""
    u = np.asarray(u, dtype=np.float64)
    with np.errstate(over="ignore"):
        return u / (1.0 + np.exp(-u))


@dataclass
class Int8Experts:
    """W8A16 expert weights in the P-int8 layout (create_weights)."""
    w13: np.ndarray   # int8 [E, 2I, H]; rows [0, I) gate (w1), [I, 2I) up (w3)
    s13: np.ndarray   # float32 [E, 2I]
    w2: np.ndarray    # int8 [E, H, I]
    s2: np.ndarray    # float32 [E, H]

    @property
    def shape(self):
        E, N2, H = self.w13.shape
        return E, H, N2 // 2

    def deq13(self, e):
        return dequantize_int8_per_channel(self.w13[e], self.s13[e])

    def deq2(self, e, rows=None):
        if rows is None:
            return dequantize_int8_per_channel(self.w2[e], self.s2[e])
        return dequantize_int8_per_channel(self.w2[e][rows], self.s2[e][rows])


# --------------------------------------------------------------------------
# W8A16 stored the moe_wna16 way (P-wna16, num_bits == 8): uint8 codes,
# one scale (and optionally one zero point) per output row
# --------------------------------------------------------------------------
def dequantize_uint8_per_channel(q, scales, zeros=None):
    """w[n, k] = (q[n, k] - z[n]) * s[n] in float64.

    Reading: without stored zero points the zero is 2^(bits-1) = 128, the
    same convention as the implicit zero 8 of the 4-bit format, so that a
    symmetric int8 code c is stored as c + 128.
    """
    q = np.asarray(q, dtype=np.float64)
    s = np.asarray(scales, dtype=np.float64).reshape(q.shape[0], 1)
    z = 128.0 if zeros is None else np.asarray(zeros, dtype=np.float64).reshape(q.shape[0], 1)
    return (q - z) * s


@dataclass
class Uint8Experts:
    """W8A16 in the P-wna16 8-bit layout: uint8 qweight, per-row scales (the
    parameter dtype's values, held as float64 here) and optional zeros."""
    qw13: np.ndarray          # uint8 [E, 2I, H]
    sc13: np.ndarray          # [E, 2I] (stored [E, 2I, 1])
    qw2: np.ndarray           # uint8 [E, H, I]
    sc2: np.ndarray           # [E, H]
    qz13: np.ndarray = None   # uint8 [E, 2I] or None (zero 128)
    qz2: np.ndarray = None    # uint8 [E, H] or None

    @property
    def shape(self):
        E, N2, H = self.qw13.shape
        return E, H, N2 // 2

    def deq13(self, e):
        return dequantize_uint8_per_channel(self.qw13[e], self.sc13[e],
                                            None if self.qz13 is None else self.qz13[e])

    def deq2(self, e, rows=None):
        z = None if self.qz2 is None else self.qz2[e]
        full = dequantize_uint8_per_channel(self.qw2[e], self.sc2[e], z)
        return full if rows is None else full[rows]


@dataclass
class Int8TensorExperts:
    """Int8 codes with one scale per expert and weight tensor (P-ct strategy
    "tensor"): w = q * s[e]."""
    w13: np.ndarray   # int8 [E, 2I, H]
    s13: np.ndarray   # [E]
    w2: np.ndarray    # int8 [E, H, I]
    s2: np.ndarray    # [E]

    @property
    def shape(self):
        E, N2, H = self.w13.shape
        return E, H, N2 // 2

    def deq13(self, e):
        return self.w13[e].astype(np.float64) * float(self.s13[e])

    def deq2(self, e, rows=None):
        w = self.w2[e] if rows is None else self.w2[e][rows]
        return w.astype(np.float64) * float(self.s2[e])


@dataclass
class Uint4Experts:
    """W4A16 expert weights in the P-wna16 layout (create_weights)."""
    qw13: np.ndarray  # uint8 [E, 2I, H/2]
    sc13: np.ndarray  # float16 [E, 2I, H/gs]
    qz13: np.ndarray  # uint8 [E, I, H/gs]   (2I rows packed two per byte)
    qw2: np.ndarray   # uint8 [E, H, I/2]
    sc2: np.ndarray   # float16 [E, H, I/gs]
    qz2: np.ndarray   # uint8 [E, H/2, I/gs]
    group_size: int
    has_zp: bool = True

    @property
    def shape(self):
        E, N2, Hh = self.qw13.shape
        return E, Hh * 2, N2 // 2

    def deq13(self, e):
        return dequantize_uint4_group(self.qw13[e], self.sc13[e], self.qz13[e],
                                      self.group_size, self.has_zp)

    def deq2(self, e, rows=None):
        full = dequantize_uint4_group(self.qw2[e], self.sc2[e], self.qz2[e],
                                      self.group_size, self.has_zp)
        return full if rows is None else full[rows]


def moe_forward(x, experts, topk_w, topk_ids, tokens=None, out_cols=None,
                apply_router_weight_on_input=False, intermediate="exact"):
    """out[t] = sum_j topk_w[t, j] * W2(e_j) . (silu(g) * u), in float64.

    g = W13(e_j)[0:I] . x[t] and u = W13(e_j)[I:2I] . x[t] use the
    dequantised weights (per-channel int8 or uint8, per-tensor int8 or
    per-group uint4).  The gate half comes first in w13, which fixes the
    SiLU-and-mul pairing.

    Reading of ``apply_router_weight_on_input`` (a name only, on the pages):
    the router weight scales the expert's input instead of its output,
    out[t] = sum_j W2(e_j) . (silu(g') * u') with g', u' computed from
    topk_w[t, j] * x[t].

    ``intermediate="bf16"`` rounds silu(g) * u to bfloat16 before the down
    projection.  Reading: the pages do not state the intermediate's
    precision; the GPU path holds it in bfloat16, the activation dtype, and
    tests of variants whose error budget that rounding dominates compare
    against this form.  The default keeps it exact.

    ``tokens`` restricts the computation to those rows (rows are independent
    once the routing is fixed); ``out_cols`` restricts the output columns
    (only those rows of W2 are then needed).  Slots with an expert id outside
    [0, E) contribute nothing.
    """
    x = np.asarray(x, dtype=np.float64)
    E, H, I = experts.shape
    ids = np.asarray(topk_ids)
    wts = np.asarray(topk_w, dtype=np.float64)
    if tokens is None:
        tokens = np.arange(x.shape[0])
    tokens = np.asarray(tokens)
    cols = np.arange(H) if out_cols is None else np.asarray(out_cols)
    out = np.zeros((tokens.size, cols.size))
    sub_ids = ids[tokens]
    sub_w = wts[tokens]
    for e in np.unique(sub_ids):
        if e < 0 or e >= E:
            continue
        rr, jj = np.nonzero(sub_ids == e)
        W13 = experts.deq13(int(e))
        W2 = experts.deq2(int(e), None if out_cols is None else cols)
        xin = x[tokens[rr]]
        if apply_router_weight_on_input:
            xin = sub_w[rr, jj][:, None] * xin
        h = xin @ W13.T
        a = silu(h[:, :I]) * h[:, I:]
        if intermediate == "bf16":
            a = round_to_bf16(a)
        y = a @ W2.T
        if apply_router_weight_on_input:
            np.add.at(out, rr, y)
        else:
            np.add.at(out, rr, sub_w[rr, jj][:, None] * y)
    return out
