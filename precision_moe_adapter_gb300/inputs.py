"""Seeded synthetic inputs for the MoE layer (shared by the tests, the
benchmark and the oracle checks).

This module only draws random numbers and lays them out; it holds none of
the layer's arithmetic (no dequantization, routing, rotation or GEMM).
Everything is generated on the host with numpy's PCG64 from an explicit
seed, so x86 and Arm hosts produce identical bytes.

Value recipes (the pages give the shapes of the workloads, not the values;
these are the plainest distributions the shapes allow):
  X            ~ N(0, 1) rounded to BF16
  dY           ~ N(0, 0.1^2) rounded to BF16   (variance 1e-2)
  Wr           ~ N(0, 0.02^2), FP32 [d, E]
  bias         uniform router: none; skewed router: -1.1 ln(pi(e) + 1) for a
               seeded permutation pi of the experts (Zipf, s = 1.1)
  INT4         nibbles uniform on [-8, 7]; BF16 scales U[0.005, 0.02]
  MXFP4        E2M1 codes uniform over all 16; E8M0 exponents U{-8..-4}
  FP8          codes = E4M3(z), z ~ N(0, 1); FP32 scale U[0.005, 0.02] per
               [128, 128] block
  S (adapter)  skew-symmetric blocks, upper triangle N(0, 0.01^2)
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

INT4, MXFP4, FP8 = 0, 1, 2
FMT_NAMES = {INT4: "int4_g32_bf16", MXFP4: "mxfp4_g32_e8m0", FP8: "fp8_e4m3_b128_f32"}

# stream ids: each tensor draws from its own seeded stream
_SID = dict(X=1, Wr=2, bias=3, w13=4, s13=5, w2=6, s2=7, S_up=8, S_down=9, dY=10,
            route=11, weights=12)


def _rng(seed: int, sid: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, _SID[sid]]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to BF16 (nearest, ties to even); returns
    uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class LayerConfig:
    """Shape and distributions of one MoE-layer workload."""
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    b: int
    fmt: int = INT4
    C: int = 16
    router: str = "uniform"          # "uniform" | "zipf"
    adapter: str = "per_expert"      # "per_expert" | "shared" | "none"
    seed: int = 0
    backward: bool = False
    notes: str = field(default="", compare=False)

    @property
    def P(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


# The workloads: a tiny parity case, three full-size layer shapes and the
# decode-sized sweep on the Kimi-K2 shape.
CONFIGS = {
    "tiny": LayerConfig("tiny", T=64, d=256, E=8, k=2, I=128, b=32, C=4, seed=0),
    "qwen3_30b_a3b": LayerConfig("qwen3_30b_a3b", T=4096, d=2048, E=128, k=8, I=768, b=32,
                                 C=16, backward=True),
    "kimi_k2": LayerConfig("kimi_k2", T=8192, d=7168, E=384, k=8, I=2048, b=64, C=32,
                           router="zipf", backward=True),
    "deepseek_v3_mxfp4": LayerConfig("deepseek_v3_mxfp4", T=16384, d=7168, E=256, k=8, I=2048,
                                     b=64, fmt=MXFP4, C=32, backward=True),
}


def decode_config(T: int, fmt: int = INT4, C: int = 32) -> LayerConfig:
    """Decode-sized forward on the Kimi-K2 shape (T in {1, 8, 64, 512})."""
    return LayerConfig(f"kimi_k2_decode_T{T}_{FMT_NAMES[fmt]}_C{C}", T=T, d=7168, E=384, k=8,
                       I=2048, b=64, fmt=fmt, C=C, router="zipf")


# ---------------------------------------------------------------- tensors

def gen_x(cfg: LayerConfig) -> np.ndarray:
    z = _rng(cfg.seed, "X").standard_normal((cfg.T, cfg.d), dtype=np.float32)
    return f32_to_bf16_bits(z)


def gen_dy(cfg: LayerConfig) -> np.ndarray:
    z = _rng(cfg.seed, "dY").standard_normal((cfg.T, cfg.d), dtype=np.float32) * np.float32(0.1)
    return f32_to_bf16_bits(z)


def gen_router(cfg: LayerConfig):
    """(Wr f32 [d, E], bias f32 [E] or None)."""
    Wr = _rng(cfg.seed, "Wr").standard_normal((cfg.d, cfg.E), dtype=np.float32) * np.float32(0.02)
    bias = None
    if cfg.router == "zipf":
        pi = _rng(cfg.seed, "bias").permutation(cfg.E)
        bias = (-1.1 * np.log(pi + 1.0)).astype(np.float32)
    return Wr, bias


def _uniform_bf16(rng, shape, lo=0.005, hi=0.02):
    out = np.empty(int(np.prod(shape)), np.uint16)
    step = 1 << 24
    for i in range(0, out.size, step):
        n = min(step, out.size - i)
        out[i:i + n] = f32_to_bf16_bits(rng.random(n, dtype=np.float32) * np.float32(hi - lo)
                                        + np.float32(lo))
    return out.reshape(shape)


def _e4m3_codes(rng, shape):
    import torch  # conversion of the Gaussian draws to the nearest E4M3 code
    out = np.empty(int(np.prod(shape)), np.uint8)
    step = 1 << 24
    for i in range(0, out.size, step):
        n = min(step, out.size - i)
        z = torch.from_numpy(rng.standard_normal(n, dtype=np.float32))
        out[i:i + n] = z.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return out.reshape(shape)


def gen_matrix(fmt: int, E: int, N: int, K: int, seed: int, qsid: str, ssid: str):
    """Quantized weights for E experts of an [N, K] linear: (q, s)."""
    rq, rs = _rng(seed, qsid), _rng(seed, ssid)
    if fmt in (INT4, MXFP4):
        q = np.frombuffer(rq.bytes(E * N * K // 2), np.uint8).reshape(E, N, K // 2).copy()
        if fmt == INT4:
            s = _uniform_bf16(rs, (E, N, K // 32))
        else:
            s = (127 + rs.integers(-8, -3, size=(E, N, K // 32))).astype(np.uint8)
        return q, s
    q = _e4m3_codes(rq, (E, N, K))
    s = (rs.random((E, N // 128, K // 128), dtype=np.float32) * np.float32(0.015)
         + np.float32(0.005)).astype(np.float32)
    return q, s


def gen_fp8_matrix_on_device(E: int, N: int, K: int, seed: int, qsid: str, ssid: str, device):
    """Full-size FP8 weights, drawn where the host recipe would take minutes
    (tens of GB of codes): codes = E4M3(z), z ~ N(0, 1) from torch's seeded
    device generator, one expert at a time; the FP32 block scales come from
    the host stream exactly as in gen_matrix.  Returns (q uint8 [E, N, K] on
    the device, s f32 [E, N/128, K/128] on the host).  The codes differ from
    gen_matrix's (another generator), the distribution is the same."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * seed + _SID[qsid])
    q = torch.empty((E, N, K), dtype=torch.uint8, device=device)
    for e in range(E):
        z = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
        q[e] = z.to(torch.float8_e4m3fn).view(torch.uint8)
    rs = _rng(seed, ssid)
    s = (rs.random((E, N // 128, K // 128), dtype=np.float32) * np.float32(0.015)
         + np.float32(0.005)).astype(np.float32)
    return q, s


def gen_weights(cfg: LayerConfig):
    """(w13, s13, w2, s2): gate rows 0..I-1 and up rows I..2I-1 of w13."""
    w13, s13 = gen_matrix(cfg.fmt, cfg.E, 2 * cfg.I, cfg.d, cfg.seed, "w13", "s13")
    w2, s2 = gen_matrix(cfg.fmt, cfg.E, cfg.d, cfg.I, cfg.seed, "w2", "s2")
    return w13, s13, w2, s2


def gen_skew(n_sets: int, dim: int, b: int, seed: int, sid: str, std: float = 0.01):
    """Skew-symmetric blocks S [n_sets, dim/b, b, b] (f32), S_ij ~ N(0, std^2)
    above the diagonal, S_ji = -S_ij, zero diagonal."""
    z = _rng(seed, sid).standard_normal((n_sets, dim // b, b, b), dtype=np.float32) * np.float32(std)
    up = np.triu(z, 1)
    return (up - np.swapaxes(up, -1, -2)).astype(np.float32)


def gen_adapter_params(cfg: LayerConfig):
    """(S_up, S_down) or (None, None) for a disabled adapter."""
    if cfg.adapter == "none":
        return None, None
    n = 1 if cfg.adapter == "shared" else cfg.E
    return (gen_skew(n, cfg.d, cfg.b, cfg.seed, "S_up"),
            gen_skew(n, cfg.I, cfg.b, cfg.seed, "S_down"))


def gen_routing(cfg: LayerConfig, skew: float = 1.1):
    """A seeded routing that does not go through the router: k distinct
    experts per token drawn with Zipf-skewed preference (skew 0 = uniform),
    and positive weights summing to one.  Returns (idx i32 [T,k], w f32 [T,k])."""
    rng = _rng(cfg.seed, "route")
    pref = -skew * np.log(rng.permutation(cfg.E) + 1.0)
    g = rng.gumbel(size=(cfg.T, cfg.E)) + pref
    idx = np.argsort(-g, axis=1, kind="stable")[:, :cfg.k].astype(np.int32)
    w = rng.random((cfg.T, cfg.k)) + 0.05
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return idx, w
