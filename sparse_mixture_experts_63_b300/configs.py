"""The five synthetic MoE-layer workloads, by shape.

T tokens, d model dim, f expert hidden dim, N routed experts, k experts per
token, fs shared-expert hidden dim (0 = none), cf capacity factor (0 = no
limit), bias_std = std of the per-expert router bias (0 = no bias).

The Mixtral-8x7B shape (8 experts, top-2) and the DeepSeek-V3 shape (256
routed experts + 1 shared, top-8) follow "MoE 分片：混合專家模型的平行化策略",
section "當前 MoE 格局"; the capacity-limited 128-expert layer follows "MoE稀疏激活
原理与工程实践", 2.2 (expert capacity) with a 128-expert router.
"""
from dataclasses import dataclass, asdict


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    f: int
    N: int
    k: int
    fs: int = 0
    cf: float = 0.0
    bias_std: float = 0.0
    dtype: str = "bf16"       # "f32" or "bf16": x and every weight
    seed: int = 0

    def as_dict(self):
        return asdict(self)

    def scaled(self, **kw) -> "MoEConfig":
        """Same config with some fields replaced (used for reduced parity cases)."""
        d = asdict(self)
        d.update(kw)
        return MoEConfig(**d)


TINY = MoEConfig("tiny", T=256, d=64, f=128, N=8, k=2, dtype="f32", seed=1)
MIXTRAL_DECODE = MoEConfig("mixtral_decode", T=32, d=4096, f=14336, N=8, k=2, seed=2)
MIXTRAL_PREFILL = MoEConfig("mixtral_prefill", T=16384, d=4096, f=14336, N=8, k=2,
                            bias_std=0.5, seed=3)
DEEPSEEK = MoEConfig("deepseek", T=8192, d=7168, f=2048, N=256, k=8, fs=2048, seed=4)
CAPACITY = MoEConfig("capacity", T=4096, d=2048, f=1408, N=128, k=2, cf=1.25,
                     bias_std=1.0, seed=5)

CONFIGS = {c.name: c for c in (TINY, MIXTRAL_DECODE, MIXTRAL_PREFILL, DEEPSEEK, CAPACITY)}
