"""Seeded synthetic inputs for the MoE layer step.

This module serves both the oracle side and the CUDA side and holds none of the
method's arithmetic: it only draws numbers.  Nothing here routes, decodes, multiplies
or activates.

Workloads (sizes and value distributions of the five configurations this library is
measured on):

  tiny            hidden 256,  inter 128,  16 experts, top-2,  1 shared, 4 tokens
  decode1         hidden 7168, inter 1536, 896 experts, top-16, 1 shared, 1 token
  decode64_zipf   as decode1, 64 tokens, bias steering expert popularity to Zipf(1.1)
  decode64_uniform  as decode1, 64 tokens, uniform routing (the pages' Quantile
                  Balancing flattens expert use, so this is the realistic batch)
  prefill4096     as decode1, 4096 tokens, uniform routing
  stacked8        8 decode1 layers, batch 1, 256 steps, RMSNorm + residual in between
  latent_decode1  the pages' LatentMoE: hidden 7168, experts in a 3584-wide latent with
                  intermediate 3072, 896 experts, top-16, 2 shared experts of width 3072
                  on the full-width input, 1 token
  latent_tiny     the same structure at hidden 256, latent 128, inter 128, 16 experts,
                  top-2, 2 shared experts, 4 tokens

Value recipe (all configurations):
  * routed experts: E2M1 nibbles uniform over all 16 codes (so packed bytes uniform over
    0..255), E8M0 scale bytes uniform over {122, ..., 126}, group 32;
  * router weight and shared-expert weights: bf16 ~ N(0, 1/fan_in) (standard deviation
    1/sqrt(fan_in): hidden for router/gate/up, inter for down);
  * correction bias: float32 U(-0.1, 0.1);
  * activations: bf16 N(0, 1);
  * LatentMoE projections: bf16 ~ N(0, 1/fan_in) (hidden for the down-projection, latent
    for the up-projection); latent RMSNorm weight float32 N(1, 0.1^2).

Expert bytes come from a counter-based generator, SplitMix64 (Steele, Lea & Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014): output i of the stream
keyed by k is mix(k + (i + 1) * 0x9E3779B97F4A7C15) with mix the SplitMix64 finaliser.
``synth/fill.cu`` implements the same definition on the device, so a 15.7 GB (or 126 GB)
expert pool is written in HBM directly while any single expert can be regenerated on the
host for the oracle.  The other tensors are small and drawn with numpy's PCG64.
"""
from dataclasses import dataclass, field, replace
import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# operand ids inside an expert record, in record order
OP_W1P, OP_W1S, OP_W2P, OP_W2S, OP_W3P, OP_W3S = range(6)
# tensor ids for the numpy-drawn tensors
T_X, T_ROUTER, T_BIAS, T_SH_GATE, T_SH_UP, T_SH_DOWN, T_ZIPF_PERM, T_ZIPF_JIT = range(8)
T_W_DOWN, T_W_UP, T_LATENT_NORM = 8, 9, 10


@dataclass(frozen=True)
class Config:
    name: str
    hidden: int
    inter: int
    n_experts: int
    topk: int
    tokens: int
    n_shared: int = 1
    layers: int = 1
    steps: int = 1
    routing: str = "uniform"          # "uniform" | "zipf"
    zipf_s: float = 1.1
    zipf_beta: float = 0.0            # bias strength, see zipf_bias()
    scale_lo: int = 122
    scale_hi: int = 126
    situ_b1: float = 4.0
    situ_b2: float = 25.0
    routed_scale: float = 1.0
    renorm: int = 1
    rms_eps: float = 1e-5
    latent: int = 0                   # > 0: a LatentMoE layer, experts in this width

    @property
    def expert_in(self):
        """Input width of the routed experts: the latent, or the hidden width."""
        return self.latent if self.latent else self.hidden

    @property
    def record_offsets(self):
        return record_offsets(self.expert_in, self.inter)

    @property
    def record_bytes(self):
        return self.record_offsets[6]

    @property
    def shared_inter(self):
        return self.inter * self.n_shared


# Bias strength for the Zipf(1.1) decode workload, from tests/golden/zipf_calibration.py:
# routing 4096 seeded tokens with this bias gives selection counts whose log-log slope
# against the popularity rank is -1.1 over ranks 17..256 (tests/golden/zipf_beta.json).
ZIPF_BETA_1P1 = 0.0551

CONFIGS = {
    "tiny": Config("tiny", 256, 128, 16, 2, 4),
    "decode1": Config("decode1", 7168, 1536, 896, 16, 1),
    "decode64_zipf": Config("decode64_zipf", 7168, 1536, 896, 16, 64, routing="zipf",
                            zipf_beta=ZIPF_BETA_1P1),
    "decode64_uniform": Config("decode64_uniform", 7168, 1536, 896, 16, 64),
    "prefill4096": Config("prefill4096", 7168, 1536, 896, 16, 4096),
    "stacked8": Config("stacked8", 7168, 1536, 896, 16, 1, layers=8, steps=256),
    "latent_decode1": Config("latent_decode1", 7168, 3072, 896, 16, 1, n_shared=2,
                             latent=3584),
    "latent_tiny": Config("latent_tiny", 256, 128, 16, 2, 4, n_shared=2, latent=128),
}


def record_offsets(H: int, I: int):
    """(w1p, w1s, w2p, w2s, w3p, w3s, total) byte offsets of the six-operand record."""
    gp, gs = I * ((H + 1) // 2), I * ((H + 31) // 32)
    dp, ds = H * ((I + 1) // 2), H * ((I + 31) // 32)
    o = [0]
    for n in (gp, gs, dp, ds, gp, gs):
        o.append(o[-1] + n)
    return o


# ----------------------------------------------------------------------------------
# SplitMix64
# ----------------------------------------------------------------------------------
def mix64(z):
    """SplitMix64 finaliser on uint64 (scalar or array); wraps modulo 2^64."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def stream(key, i):
    """Output i (0-based, uint64 array) of the SplitMix64 stream keyed by ``key``."""
    i = np.asarray(i, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + (i + np.uint64(1)) * GOLDEN)


def operand_key(seed: int, layer: int, expert: int, op: int) -> np.uint64:
    """Stream key of one operand of one expert of one layer."""
    with np.errstate(over="ignore"):
        k = mix64(np.uint64(seed) + GOLDEN)
        k = mix64(k + np.uint64(layer))
        k = mix64(k + np.uint64(expert) * np.uint64(8) + np.uint64(op))
    return np.uint64(k)


def packed_bytes(key, nbytes: int) -> np.ndarray:
    """nbytes uniform bytes: byte b is byte (b % 8) (little-endian) of stream output b/8."""
    words = stream(key, np.arange((nbytes + 7) // 8, dtype=np.uint64))
    return words.view(np.uint8)[:nbytes].copy()


def scale_bytes(key, nbytes: int, lo: int, hi: int) -> np.ndarray:
    """nbytes scale bytes uniform over {lo..hi}: lo + floor((output_b >> 32) * n / 2^32)."""
    h = stream(key, np.arange(nbytes, dtype=np.uint64)) >> np.uint64(32)
    with np.errstate(over="ignore"):
        v = (h * np.uint64(hi - lo + 1)) >> np.uint64(32)
    return (v + np.uint64(lo)).astype(np.uint8)


def expert_record(cfg: Config, seed: int, layer: int, expert: int) -> np.ndarray:
    """The full byte record of one routed expert (uint8 [record_bytes])."""
    off = cfg.record_offsets
    rec = np.empty(off[6], dtype=np.uint8)
    for op in range(6):
        n = off[op + 1] - off[op]
        key = operand_key(seed, layer, expert, op)
        if op in (OP_W1P, OP_W2P, OP_W3P):
            rec[off[op]:off[op + 1]] = packed_bytes(key, n)
        else:
            rec[off[op]:off[op + 1]] = scale_bytes(key, n, cfg.scale_lo, cfg.scale_hi)
    return rec


def all_experts(cfg: Config, seed: int, layer: int = 0) -> np.ndarray:
    """Every routed expert of a layer, uint8 [E][record_bytes] (small configs only)."""
    return np.stack([expert_record(cfg, seed, layer, e) for e in range(cfg.n_experts)])


# ----------------------------------------------------------------------------------
# numpy-drawn tensors
# ----------------------------------------------------------------------------------
def _rng(seed: int, layer: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, tensor])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, nearest-even (input generation only)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def normal_bf16(seed, layer, tensor, shape, std) -> np.ndarray:
    g = _rng(seed, layer, tensor).standard_normal(shape, dtype=np.float32)
    return to_bf16_bits(g * np.float32(std))


def activations(cfg: Config, seed: int, tokens: int = None) -> np.ndarray:
    """Layer input x, bf16 bits [T][H], N(0,1)."""
    T = cfg.tokens if tokens is None else tokens
    return normal_bf16(seed, 0, T_X, (T, cfg.hidden), 1.0)


def zipf_ranks(cfg: Config, seed: int, layer: int) -> np.ndarray:
    """Popularity rank (1 = most popular) of every expert: a seeded permutation."""
    E = cfg.n_experts
    perm = _rng(seed, layer, T_ZIPF_PERM).permutation(E)
    rank = np.empty(E, dtype=np.int64)
    rank[perm] = np.arange(1, E + 1)
    return rank


def zipf_bias(cfg: Config, seed: int, layer: int) -> np.ndarray:
    """Correction bias making expert popularity follow Zipf(s): a seeded permutation
    ranks the experts, bias_e = beta ln(p_e / p_max) + U(-0.1, 0.1), p_e ~ rank^-s."""
    E = cfg.n_experts
    rank = zipf_ranks(cfg, seed, layer)
    logp = -cfg.zipf_s * np.log(rank.astype(np.float64))
    jit = _rng(seed, layer, T_ZIPF_JIT).uniform(-0.1, 0.1, E)
    return (cfg.zipf_beta * logp + jit).astype(np.float32)


def layer_weights(cfg: Config, seed: int, layer: int = 0) -> dict:
    """Router weight, bias and shared-expert weights of one layer (numpy arrays)."""
    H, I, E = cfg.hidden, cfg.inter, cfg.n_experts
    SI = cfg.shared_inter
    if cfg.routing == "zipf":
        bias = zipf_bias(cfg, seed, layer)
    else:
        bias = _rng(seed, layer, T_BIAS).uniform(-0.1, 0.1, E).astype(np.float32)
    out = {
        "wr": normal_bf16(seed, layer, T_ROUTER, (E, H), 1.0 / math.sqrt(H)),
        "bias": bias,
    }
    if cfg.n_shared > 0:
        out["sh_gate"] = normal_bf16(seed, layer, T_SH_GATE, (SI, H), 1.0 / math.sqrt(H))
        out["sh_up"] = normal_bf16(seed, layer, T_SH_UP, (SI, H), 1.0 / math.sqrt(H))
        out["sh_down"] = normal_bf16(seed, layer, T_SH_DOWN, (H, SI), 1.0 / math.sqrt(SI))
    if cfg.latent:
        L = cfg.latent
        out["w_down"] = normal_bf16(seed, layer, T_W_DOWN, (L, H), 1.0 / math.sqrt(H))
        out["w_up"] = normal_bf16(seed, layer, T_W_UP, (H, L), 1.0 / math.sqrt(L))
        out["norm_w"] = (1.0 + 0.1 * _rng(seed, layer, T_LATENT_NORM).standard_normal(
            L, dtype=np.float32)).astype(np.float32)
    return out


def config(name: str, **overrides) -> Config:
    cfg = CONFIGS[name]
    return replace(cfg, **overrides) if overrides else cfg
