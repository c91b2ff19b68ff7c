"""Seeded synthetic workloads for the Hadamard route.

This module only draws inputs: shapes, value distributions and outlier
structure of the prompt-processing workloads (the pages measure whole models
on real prompts, which are not available, so these synthetic inputs stand in
for them).  It holds none of the method's arithmetic: no rotation, no
quantization, no dot products.  Both the CUDA path and the CPU oracle consume
exactly these arrays.

Generator: numpy PCG64 seeded with ``[seed, config_id, tensor_id]``.  Values
are drawn in fp32; bf16 inputs are the fp32 draws rounded to nearest even
(returned as uint16 bit patterns).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# config ids (part of every seed)
CFG_TINY, CFG_ATTN, CFG_FFN, CFG_MOE, CFG_LONG, CFG_TEST = 0, 1, 2, 3, 4, 9


def rng(seed: int, config_id: int, tensor_id: int) -> np.random.Generator:
    return np.random.default_rng([seed, config_id, tensor_id])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even), returned as uint16 bits.  Inputs are finite."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def outlier_channels(K: int, frac: float, seed: int, config_id: int, tensor_id: int) -> np.ndarray:
    """round(frac*K) distinct channel indices, fixed for every token."""
    n = int(round(frac * K))
    if n == 0:
        return np.zeros(0, np.int64)
    return np.sort(rng(seed, config_id, tensor_id + 1000).choice(K, size=n, replace=False))


def act_normal_outliers(M: int, K: int, frac: float, scale: float, seed: int,
                        config_id: int, tensor_id: int) -> np.ndarray:
    """fp32 N(0,1) [M][K] with a fixed set of outlier channels multiplied by ``scale``."""
    x = rng(seed, config_id, tensor_id).standard_normal((M, K), dtype=np.float32)
    ch = outlier_channels(K, frac, seed, config_id, tensor_id)
    if ch.size:
        x[:, ch] *= np.float32(scale)
    return x


def act_student_t(M: int, K: int, nu: float, scale: float, seed: int, config_id: int,
                  tensor_id: int) -> np.ndarray:
    x = rng(seed, config_id, tensor_id).standard_t(nu, size=(M, K)).astype(np.float32)
    return x * np.float32(scale)


def weights_normal(N: int, K: int, sigma: float, seed: int, config_id: int,
                   tensor_id: int) -> np.ndarray:
    w = rng(seed, config_id, tensor_id).standard_normal((N, K), dtype=np.float32)
    return w * np.float32(sigma)


# --------------------------------------------------------------------------
# projections and configurations
# --------------------------------------------------------------------------
@dataclass
class Projection:
    """One (quantize activations -> GEMM) step: y[M][N] = x[M][K] . W[N][K]^T."""
    name: str
    K: int
    N: int
    act: str            # "normal_outliers" | "student_t"
    act_frac: float = 0.0
    act_scale: float = 1.0
    nu: float = 4.0
    sigma: float = 0.02
    tensor_id: int = 0  # activations use tensor_id, weights tensor_id + 1

    def activations(self, M: int, seed: int, config_id: int, bf16: bool = True,
                    tensor_offset: int = 0) -> np.ndarray:
        tid = self.tensor_id + tensor_offset
        if self.act == "student_t":
            x = act_student_t(M, self.K, self.nu, self.act_scale, seed, config_id, tid)
        else:
            x = act_normal_outliers(M, self.K, self.act_frac, self.act_scale, seed, config_id, tid)
        return f32_to_bf16_bits(x) if bf16 else x

    def weights(self, seed: int, config_id: int) -> np.ndarray:
        return weights_normal(self.N, self.K, self.sigma, seed, config_id, self.tensor_id + 1)


ATTN = Projection("attn", K=5120, N=5120, act="normal_outliers", act_frac=0.005,
                  act_scale=30.0, tensor_id=10)
FFN_GATE_UP = Projection("ffn_gate_up", K=5120, N=2 * 17408, act="student_t", act_scale=0.5,
                         tensor_id=20)
FFN_DOWN = Projection("ffn_down", K=17408, N=5120, act="student_t", act_scale=0.5, tensor_id=30)

# the long-prompt sweep uses the same chain with N(0,1) + 0.5% x30 activations
LONG_ATTN = Projection("attn", K=5120, N=5120, act="normal_outliers", act_frac=0.005,
                       act_scale=30.0, tensor_id=40)
LONG_GATE_UP = Projection("ffn_gate_up", K=5120, N=2 * 17408, act="normal_outliers",
                          act_frac=0.005, act_scale=30.0, tensor_id=50)
LONG_DOWN = Projection("ffn_down", K=17408, N=5120, act="normal_outliers", act_frac=0.005,
                       act_scale=30.0, tensor_id=60)


@dataclass
class DenseConfig:
    name: str
    config_id: int
    M: int
    chain: list = field(default_factory=list)
    bf16: bool = True
    micro_batch: int = 0   # 0 = one batch of M tokens


TINY = DenseConfig("tiny", CFG_TINY, M=64, bf16=False, chain=[
    Projection("tiny", K=256, N=256, act="normal_outliers", act_frac=0.01, act_scale=20.0,
               tensor_id=0)])

PP512_ATTN = DenseConfig("pp512_attn", CFG_ATTN, M=512, chain=[ATTN])
PP512_FFN = DenseConfig("pp512_ffn", CFG_FFN, M=512, chain=[FFN_GATE_UP, FFN_DOWN])
# the pp512 GEMM chain: attention projection then the dense FFN
PP512_CHAIN = DenseConfig("pp512_chain", CFG_FFN, M=512, chain=[ATTN, FFN_GATE_UP, FFN_DOWN])


def long_config(M: int) -> DenseConfig:
    return DenseConfig(f"long_{M}", CFG_LONG, M=M, micro_batch=1024,
                       chain=[LONG_ATTN, LONG_GATE_UP, LONG_DOWN])


LONG_MS = (1024, 2048, 8192, 16384)


def chain_config_id(cfg: DenseConfig, proj: Projection) -> int:
    """The attention projection of the chain draws from the attention config's stream."""
    if cfg.name == "pp512_chain" and proj is ATTN:
        return CFG_ATTN
    return cfg.config_id


# --------------------------------------------------------------------------
# MoE experts
# --------------------------------------------------------------------------
@dataclass
class MoEConfig:
    name: str = "moe"
    config_id: int = CFG_MOE
    T: int = 1024          # tokens in the micro-batch
    hidden: int = 2048
    ffn: int = 768
    E: int = 128
    top_k: int = 8
    act_frac: float = 0.005
    act_scale: float = 30.0
    sigma: float = 0.02


MOE = MoEConfig()


def moe_logits(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    """Router logits [T][E] fp32, U(0,1)."""
    return rng(seed, cfg.config_id, 0).random((cfg.T, cfg.E), dtype=np.float32)


def moe_routing(cfg: MoEConfig, seed: int = 0):
    """Top-k experts per token from U(0,1) logits, grouped by expert.

    Softmax is monotonic, so the top-k of the softmax are the top-k logits;
    ties go to the lower expert id.  Returns (row_idx [T*k] int32: the token of
    each grouped row, expert_off [E+1] int32, expert_of_row [T*k] int32).
    Rows are grouped by expert, and within an expert kept in token order."""
    logits = moe_logits(cfg, seed)
    # stable sort on -logit keeps the lower id first among equal logits
    order = np.argsort(-logits, axis=1, kind="stable")[:, :cfg.top_k]
    tok = np.repeat(np.arange(cfg.T, dtype=np.int64), cfg.top_k)
    exp = order.reshape(-1).astype(np.int64)
    g = np.lexsort((tok, exp))       # by expert, then token
    row_idx = tok[g].astype(np.int32)
    expert_of_row = exp[g].astype(np.int32)
    counts = np.bincount(exp, minlength=cfg.E)
    off = np.zeros(cfg.E + 1, np.int32)
    off[1:] = np.cumsum(counts)
    return row_idx, off, expert_of_row


def moe_inputs(cfg: MoEConfig, seed: int = 0):
    """Activations and fp32 expert weights of one MoE micro-batch.

    x_gate_up: bf16 bits [T][hidden] (N(0,1) + outlier channels)
    x_down:    bf16 bits [T*k][ffn] (an independent draw of the same law; the
               SwiGLU that would produce it is outside the path)
    w_gate_up: fp32 [E][2*ffn][hidden];  w_down: fp32 [E][hidden][ffn]"""
    x_gu = f32_to_bf16_bits(act_normal_outliers(cfg.T, cfg.hidden, cfg.act_frac, cfg.act_scale,
                                                 seed, cfg.config_id, 1))
    R = cfg.T * cfg.top_k
    x_dn = f32_to_bf16_bits(act_normal_outliers(R, cfg.ffn, cfg.act_frac, cfg.act_scale,
                                                seed, cfg.config_id, 2))
    return x_gu, x_dn


def moe_weights(cfg: MoEConfig, seed: int = 0):
    w_gu = weights_normal(cfg.E * 2 * cfg.ffn, cfg.hidden, cfg.sigma, seed, cfg.config_id, 3)
    w_dn = weights_normal(cfg.E * cfg.hidden, cfg.ffn, cfg.sigma, seed, cfg.config_id, 4)
    return (w_gu.reshape(cfg.E, 2 * cfg.ffn, cfg.hidden),
            w_dn.reshape(cfg.E, cfg.hidden, cfg.ffn))
