"""The five workloads: shapes, masks, dtypes and seeds (workload n uses seed 1000 + n)."""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Config:
    name: str
    batch: int
    n_heads: int
    n_kv: int
    d: int
    Tq: int
    Tk: int                       # key/value cache length (Tk_max when lengths vary)
    dtype: str                    # 'f32' or 'bf16'
    causal: bool = True
    window: int = 0
    sink: bool = False
    k_len_range: tuple | None = None   # (lo, hi) inclusive per-sequence lengths, else all Tk
    q_block: int = 128
    k_block: int = 64
    planted_fraction: float = 0.0
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def g(self) -> int:
        return self.n_heads // self.n_kv


CONFIGS = {
    1: Config("fp32 tiny GQA, prefill T=40 and token-by-token decode", 1, 8, 2, 16, 40, 40,
              "f32", seed=1001),
    2: Config("bf16 dense causal GQA prefill B2 H32 Hkv8 d128 T8192", 2, 32, 8, 128, 8192,
              8192, "bf16", seed=1002),
    3: Config("bf16 KV-cache decode B64 H32 Hkv8 d128 Tk<=32768 (lengths U[16384,32768]), "
              "Tq=1 and a Tq=512 chunk", 64, 32, 8, 128, 1, 32768, "bf16",
              k_len_range=(16384, 32768), seed=1003, extra={"chunk_Tq": 512}),
    4: Config("bf16 sliding window 1024 + sink, B1 H16 Hkv8 d256 T32768 (and full causal)",
              1, 16, 8, 256, 32768, 32768, "bf16", window=1024, sink=True, seed=1004),
    5: Config("bf16 block-sparse prefill B1 H32 Hkv8 d128 T131072, key block 64, query "
              "block 128, 5% planted outlier blocks", 1, 32, 8, 128, 131072, 131072, "bf16",
              planted_fraction=0.05, seed=1005,
              extra={"lambda_radius": 3.0}),
}


def get_config(n: int) -> Config:
    return CONFIGS[n]
