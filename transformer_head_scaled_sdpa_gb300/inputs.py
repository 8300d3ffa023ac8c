"""Seeded synthetic inputs for the attention workloads.

This module is shared by the CUDA path's tests and benchmark and by the oracle
checks.  It holds no attention arithmetic: it only draws random numbers and
casts them, so both sides of a parity test receive the same bits.

Recipe (one CPU ``torch.Generator`` per workload, seed = 1000 + the
workload's index in ``WORKLOADS``): draw Q, then K, then V as float32 N(0, 1)
samples of shape [B, L, H, d_k], multiply by the workload's input scale
(1.0, or 0.5 for the GPT-3-like workload: exact in float32), and cast with
round-to-nearest-even to the workload's dtype; under key padding then draw
``key_lens`` uniformly from [len_lo, len_hi] as int32.

The shapes stand in for the pages' models, whose data (WMT14, GPT-3's corpus)
are not available: the base Transformer (d_model 512, 8 heads of d_k = 64;
"Attention Is All You Need", Sections 3.1 and 3.2.2, and the cookipedia
article's encoder/decoder sections), the big model's 16 heads, GPT-3's
96 heads of d_k = 128 at a 2048-token context (formula page
transformer-attention, section 起源 and 応用), and the cookipedia toy model
(d_model 6, 2 heads, source length 8, target length 4; section トイモデル).
"""
from __future__ import annotations

import dataclasses

import torch

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_KEY_PADDING = 2
MASK_CAUSAL_KEY_PADDING = 3  # both masks (a decoder over padded sequences)

MASK_NAMES = {MASK_NONE: "none", MASK_CAUSAL: "causal", MASK_KEY_PADDING: "key_padding",
              MASK_CAUSAL_KEY_PADDING: "causal_key_padding"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    d_k: int
    Lq: int
    Lk: int
    mask_kind: int
    dtype: torch.dtype
    input_scale: float = 1.0
    len_lo: int = 0          # key padding: key_lens ~ U[len_lo, len_hi]
    len_hi: int = 0
    note: str = ""

    @property
    def seed(self) -> int:
        return 1000 + WORKLOAD_INDEX[self.name]

    def flops(self, key_lens=None) -> float:
        """Nominal 4*B*H*Lq*Lk*d_k, halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.Lq * self.Lk * self.d_k
        return f / 2 if self.mask_kind == MASK_CAUSAL else f


WORKLOADS = [
    Workload("toy_cross_f32", 1, 2, 3, 4, 8, MASK_NONE, torch.float32,
             note="cookipedia toy model: d_model 6, 2 heads, target 4, source 8"),
    Workload("base_encoder_self", 32, 8, 64, 128, 128, MASK_NONE, torch.bfloat16,
             note="base model encoder self-attention"),
    Workload("base_decoder_causal", 32, 8, 64, 512, 512, MASK_CAUSAL, torch.bfloat16,
             note="base model decoder masked self-attention"),
    Workload("base_cross_keypad", 64, 8, 64, 256, 512, MASK_KEY_PADDING, torch.bfloat16,
             len_lo=256, len_hi=512,
             note="base model cross-attention, encoder key padding"),
    Workload("gpt3_causal", 4, 96, 128, 2048, 2048, MASK_CAUSAL, torch.bfloat16,
             input_scale=0.5, note="GPT-3-like: 96 heads, d_k 128, 2048 context"),
    # supplementary long-sequence rows at d_k = 64
    Workload("big16_L2048", 8, 16, 64, 2048, 2048, MASK_NONE, torch.bfloat16,
             note="big model head count, L 2048"),
    Workload("big16_L2048_causal", 8, 16, 64, 2048, 2048, MASK_CAUSAL, torch.bfloat16),
    Workload("base8_L4096", 16, 8, 64, 4096, 4096, MASK_NONE, torch.bfloat16),
    Workload("base8_L4096_causal", 16, 8, 64, 4096, 4096, MASK_CAUSAL, torch.bfloat16),
    # one sequence of the GPT-3-like shape (150 MB of inputs, still above L2):
    # the small case for detailed profiler captures
    Workload("gpt3_causal_b1", 1, 96, 128, 2048, 2048, MASK_CAUSAL, torch.bfloat16,
             input_scale=0.5, note="GPT-3-like, one sequence"),
    # heads of 256 features (the pages fix no head width: keys of d_k, values
    # of d_v), 16 heads at L 2048: the wide kernel's measurement rows
    Workload("d256_L2048", 4, 16, 256, 2048, 2048, MASK_NONE, torch.bfloat16,
             note="16 heads of d_k 256, L 2048"),
    Workload("d256_L2048_causal", 4, 16, 256, 2048, 2048, MASK_CAUSAL, torch.bfloat16,
             note="16 heads of d_k 256, L 2048, causal"),
]
WORKLOAD_INDEX = {w.name: i for i, w in enumerate(WORKLOADS)}
BY_NAME = {w.name: w for w in WORKLOADS}


def generate(w: Workload, seed: int | None = None, batch: slice | None = None):
    """Return dict(q, k, v, key_lens) on the CPU for workload ``w``.

    ``batch`` selects sequences after drawing (so a slice sees exactly the
    values the full draw has).  ``key_lens`` is None unless key padding.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    shape_q = (w.B, w.Lq, w.H, w.d_k)
    shape_kv = (w.B, w.Lk, w.H, w.d_k)
    out = {}
    for name, shape in (("q", shape_q), ("k", shape_kv), ("v", shape_kv)):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if w.input_scale != 1.0:
            x.mul_(w.input_scale)
        out[name] = x.to(w.dtype)
    key_lens = None
    if w.mask_kind & MASK_KEY_PADDING:
        key_lens = torch.randint(w.len_lo, w.len_hi + 1, (w.B,), generator=g,
                                 dtype=torch.int64).to(torch.int32)
    out["key_lens"] = key_lens
    if batch is not None:
        for name in ("q", "k", "v"):
            out[name] = out[name][batch].contiguous()
        if key_lens is not None:
            out["key_lens"] = key_lens[batch].contiguous()
    return out


def random_case(seed: int, B: int, H: int, Lq: int, Lk: int, d_k: int,
                dtype=torch.bfloat16, input_scale: float = 1.0,
                key_lens_range: tuple[int, int] | None = None, d_v: int | None = None):
    """Ad-hoc seeded case with the same recipe (for parity sweeps); v rows have
    width ``d_v`` (default d_k)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {}
    for name, L, w in (("q", Lq, d_k), ("k", Lk, d_k), ("v", Lk, d_v or d_k)):
        x = torch.randn((B, L, H, w), generator=g, dtype=torch.float32)
        if input_scale != 1.0:
            x.mul_(input_scale)
        out[name] = x.to(dtype)
    out["key_lens"] = None
    if key_lens_range is not None:
        lo, hi = key_lens_range
        out["key_lens"] = torch.randint(lo, hi + 1, (B,), generator=g,
                                        dtype=torch.int64).to(torch.int32)
    return out


# ---------------------------------------------------------------------------
# decode steps: one new query per sequence against a key/value cache
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One decode step of a batch of `sources` inputs with `beams` beams each
    (the pages' beam search keeps 4): B = sources * beams sequences, each with
    its own cache of capacity Lk; the beams of a source share one cache length,
    drawn uniformly from [len_lo, len_hi]."""
    name: str
    sources: int
    beams: int
    H: int
    d_k: int
    Lk: int
    len_lo: int
    len_hi: int
    input_scale: float = 1.0
    note: str = ""

    @property
    def B(self) -> int:
        return self.sources * self.beams

    @property
    def seed(self) -> int:
        return 2000 + DECODE_INDEX[self.name]


DECODE_WORKLOADS = [
    DecodeWorkload("base_decode", 32, 4, 8, 64, 256, 16, 256,
                   note="base model decoder self-attention, 32 sentences x beam 4"),
    DecodeWorkload("gpt3_decode", 4, 4, 96, 128, 2048, 1024, 2048, input_scale=0.5,
                   note="GPT-3-like, 4 prompts x beam 4, 2048 context"),
    DecodeWorkload("gpt3_decode_b1", 1, 4, 96, 128, 2048, 1024, 2048, input_scale=0.5,
                   note="GPT-3-like, one prompt x beam 4"),
]
DECODE_INDEX = {w.name: i for i, w in enumerate(DECODE_WORKLOADS)}
DECODE_BY_NAME = {w.name: w for w in DECODE_WORKLOADS}


def generate_decode(w: DecodeWorkload, seed: int | None = None):
    """Return dict(q [B, H, d], k_cache, v_cache [B, Lk, H, d], cache_lens [B]
    int32) on the CPU.  Same recipe as `generate`: q, then K, then V as
    float32 N(0, 1) times the input scale, cast to bf16; then one length per
    source, repeated for its beams."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    out = {}
    for name, shape in (("q", (w.B, w.H, w.d_k)), ("k_cache", (w.B, w.Lk, w.H, w.d_k)),
                        ("v_cache", (w.B, w.Lk, w.H, w.d_k))):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if w.input_scale != 1.0:
            x.mul_(w.input_scale)
        out[name] = x.to(torch.bfloat16)
    per_source = torch.randint(w.len_lo, w.len_hi + 1, (w.sources,), generator=g,
                               dtype=torch.int64)
    out["cache_lens"] = per_source.repeat_interleave(w.beams).to(torch.int32)
    return out



# ---------------------------------------------------------------------------
# the multi-head attention layer: projections around the attention
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class LayerWorkload:
    """One multi-head attention layer ("Attention Is All You Need", section
    3.2.2): queries from x [B, Lq, d_model], keys and values from x itself
    (self-attention, ``cross`` False, Lk = Lq) or from an encoder memory
    [B, Lk, d_model] (cross-attention); H heads of width d_k (d_v = d_k).
    Random weights (no trained ones exist here)."""
    name: str
    B: int
    Lq: int
    Lk: int
    d_model: int
    H: int
    d_k: int
    mask_kind: int
    cross: bool = False
    len_lo: int = 0          # key padding: key_lens ~ U[len_lo, len_hi]
    len_hi: int = 0
    note: str = ""

    @property
    def seed(self) -> int:
        return 3000 + LAYER_INDEX[self.name]

    def flops(self, key_lens=None) -> float:
        """Algorithmic flops: the Q, K, V and output projections (2 per
        multiply-add) plus the attention's 4*d_k per visible (query, key) pair."""
        hd = self.H * self.d_k
        proj = 2.0 * self.B * (self.Lq * self.d_model * hd + self.Lk * self.d_model * 2 * hd +
                               self.Lq * hd * self.d_model)
        if self.mask_kind == MASK_CAUSAL:
            pairs = self.B * self.H * self.Lq * (self.Lq + 1) / 2
        elif self.mask_kind & MASK_KEY_PADDING and key_lens is not None:
            lens = key_lens.clamp(0, self.Lk).to(torch.int64)
            if self.mask_kind & MASK_CAUSAL:
                i = torch.arange(self.Lq, dtype=torch.int64)
                pairs = float(self.H * torch.minimum(i[None, :] + 1, lens[:, None]).sum().item())
            else:
                pairs = float(self.H * self.Lq * lens.sum().item())
        else:
            pairs = float(self.B * self.H * self.Lq * self.Lk)
        return proj + 4.0 * self.d_k * pairs


LAYER_WORKLOADS = [
    LayerWorkload("base_layer_decoder", 32, 128, 128, 512, 8, 64, MASK_CAUSAL,
                  note="base model (d_model 512, 8 heads of 64): decoder self-attention layer"),
    LayerWorkload("base_layer_cross", 32, 128, 160, 512, 8, 64, MASK_KEY_PADDING, cross=True,
                  len_lo=64, len_hi=160,
                  note="base model: encoder-decoder attention over padded encoder outputs"),
    LayerWorkload("gpt3_layer", 4, 2048, 2048, 12288, 96, 128, MASK_CAUSAL,
                  note="GPT-3-like: d_model 12288, 96 heads of 128, 2048 context, causal"),
    LayerWorkload("gpt3_layer_b1", 1, 2048, 2048, 12288, 96, 128, MASK_CAUSAL,
                  note="GPT-3-like, one sequence"),
]
LAYER_INDEX = {w.name: i for i, w in enumerate(LAYER_WORKLOADS)}
LAYER_BY_NAME = {w.name: w for w in LAYER_WORKLOADS}


def generate_layer(w: LayerWorkload, seed: int | None = None):
    """Return dict(x [B, Lq, d_model], mem [B, Lk, d_model] or None, w_qkv
    [d_model, 3 H d_k], w_o [H d_k, d_model], key_lens [B] int32 or None) in
    bf16 on the CPU.  Draw order: x, (mem), w_qkv, w_o, (key_lens).  x and mem
    are N(0, 1); w_qkv is N(0, 1/d_model) and w_o N(0, 1/(H d_k)) (Xavier-like:
    the projections come out near N(0, 1) again).  w_qkv's columns are W^Q,
    W^K, W^V in that order, head h at columns h d_k .. h d_k + d_k - 1 of each."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    hd = w.H * w.d_k

    def draw(shape, std=1.0):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16)

    out = {"x": draw((w.B, w.Lq, w.d_model))}
    out["mem"] = draw((w.B, w.Lk, w.d_model)) if w.cross else None
    out["w_qkv"] = draw((w.d_model, 3 * hd), w.d_model ** -0.5)
    out["w_o"] = draw((hd, w.d_model), hd ** -0.5)
    out["key_lens"] = None
    if w.mask_kind & MASK_KEY_PADDING:
        out["key_lens"] = torch.randint(w.len_lo, w.len_hi + 1, (w.B,), generator=g,
                                        dtype=torch.int64).to(torch.int32)
    return out
