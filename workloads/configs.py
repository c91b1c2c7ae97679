"""The synthetic workloads this library is measured and checked on.

Each entry restates one workload: the projection shape, the token counts, the
envelope rank ell, and how signs, scales and activations are drawn (see
workloads.generators for the draw recipe and seeds).
"""

from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Projection:
    name: str
    N: int
    M: int
    R: int
    ell: int
    seed: int
    sign_mode: str = "bernoulli"
    scale_mode: str = "lordba"


@dataclass(frozen=True)
class Workload:
    key: str
    title: str
    projections: tuple
    tokens: tuple
    outlier_scale: float = 0.0
    x_seed_offset: int = 0
    n_adapters: int = 0          # > 0 only for the multi-adapter workload
    routing_seed: int = 0
    regime: str = "decode"       # "decode" or "prefill"
    extra: dict = field(default_factory=dict)


TINY = Workload(
    key="tiny",
    title="tiny double-binary matmul N=M=256 R=32 ell=1",
    projections=(Projection("tiny", 256, 256, 32, 1, 0, "gauss", "tiny"),),
    tokens=(1, 8),
)

ADAPTER_4K = Workload(
    key="adapter4k",
    title="LoRDBA unmerged adapter branch, N=M=4096 R=64 ell=1",
    projections=(Projection("adapter", 4096, 4096, 64, 1, 2000),),
    tokens=(1, 4, 16),
)

DBF_1P5 = Workload(
    key="dbf1p5",
    title="DBF full-weight replacement at 1.5 bits/weight, N=M=4096 R=3072 ell=1",
    projections=(Projection("dbf", 4096, 4096, 3072, 1, 3000),),
    tokens=(1, 8),
    outlier_scale=20.0,
)

DBF_MLP = Workload(
    key="dbfmlp",
    title="DBF MLP layer in prefill, up 14336x4096 and down 4096x14336, R=5013 ell=2, T=2048",
    projections=(Projection("up", 14336, 4096, 5013, 2, 4000),
                 Projection("down", 4096, 14336, 5013, 2, 4001)),
    tokens=(2048,),
    regime="prefill",
)

MULTI_ADAPTER = Workload(
    key="multiadapter",
    title="multi-adapter serving, 64 adapters N=M=4096 R=32 ell=2, 256 tokens",
    projections=tuple(Projection(f"adapter{a}", 4096, 4096, 32, 2, 5000 + a)
                      for a in range(64)),
    tokens=(256,),
    n_adapters=64,
    routing_seed=5999,
)

WORKLOADS = {w.key: w for w in (TINY, ADAPTER_4K, DBF_1P5, DBF_MLP, MULTI_ADAPTER)}


def algorithmic_bytes(N: int, M: int, R: int, ell: int, T: int, accumulate: bool = False) -> int:
    """Bytes a call must move at least once: sign bits, fp16 scales, x and y.

    R(N+M)/8 for the two sign matrices at one bit per entry (no padding),
    2*ell*(N+R+M) for the fp16 scales, 2*T*M for bf16 x, 2*T*N for bf16 y,
    plus 2*T*N more when y is read back for accumulation.
    """
    b = (R * (N + M)) // 8 + 2 * ell * (N + R + M) + 2 * T * M + 2 * T * N
    if accumulate:
        b += 2 * T * N
    return b


def flops(N: int, M: int, R: int, ell: int, T: int) -> int:
    """Multiply-add count of the two sign contractions, 2*T*ell*R*(N+M)."""
    return 2 * T * ell * R * (N + M)
