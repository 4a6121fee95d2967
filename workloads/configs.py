"""Synthetic workloads for the blockwise-FP8 routed-MoE layer.

Shapes and value distributions of the five workload families:

* ``tiny``          T=4, H=256, E=8, top-2, I=128 (the small parity case)
* ``olmoe_decode``  T in {1, 8}, H=2048, E=64, top-8, I=1024 (OLMoE-1B-7B shape,
                    the Trochilus page's model; memory-bound grouped GEMV)
* ``olmoe_prefill`` T in {512, 2048}, same shape, router bias ~N(0, 0.5) for
                    skewed expert loads (the Trochilus page's 512/2048-token prompts)
* ``wide_decode``   T in {1, 16, 64}, H=4096, E=384, top-6, I=2048 (the 384-expert,
                    top-6 routing of the DeepSeek-V4.1-Flash post)
* ``large_prefill`` T=4096, H=6144, E=512, top-12, I=2048, router bias ~N(0, 1):
                    heavy imbalance with experts that receive no token
* ``dense_ffn``     T in {8, 2048}, H=2048, one expert, top-1, I=8192: a dense
                    (or shared-expert) SwiGLU FFN in the same blockwise-FP8
                    format (dragon.c, "Precision": the per-sub-block dense
                    branches are e4m3 with 128x128 f32 block scales too); with
                    one expert the router gives every token weight 1

All families draw x ~ N(0,1) rounded to bf16, router W ~ N(0, 0.02) in f32, and
expert weights ~ N(0, 0.02) quantised to e4m3 with one f32 scale per 128x128
block (the dragon.c page, "Precision").  Seeds: tiny 1, olmoe_decode 2,
olmoe_prefill 3, wide_decode 4, large_prefill 5, dense_ffn 6; the activations of a T-token
batch use seed*1000 + T so that each T has its own batch.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Family:
    name: str
    hidden: int        # H
    n_experts: int     # E
    top_k: int         # k
    inter: int         # I (expert FFN width)
    seed: int
    tokens: tuple      # the T values this family is run at
    bias_std: float | None = None  # router bias ~N(0, bias_std) or no bias
    w_std: float = 0.02
    router_std: float = 0.02

    def x_seed(self, T: int) -> int:
        return self.seed * 1000 + T

    @property
    def expert_bytes(self) -> int:
        """e4m3 codes + f32 block scales of one expert (w13 and w2)."""
        H, I = self.hidden, self.inter
        return 3 * H * I + 4 * ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128))


FAMILIES = {
    "tiny": Family("tiny", 256, 8, 2, 128, 1, (4,)),
    "olmoe_decode": Family("olmoe_decode", 2048, 64, 8, 1024, 2, (1, 8)),
    "olmoe_prefill": Family("olmoe_prefill", 2048, 64, 8, 1024, 3, (512, 2048), bias_std=0.5),
    "wide_decode": Family("wide_decode", 4096, 384, 6, 2048, 4, (1, 16, 64)),
    "large_prefill": Family("large_prefill", 6144, 512, 12, 2048, 5, (4096,), bias_std=1.0),
    "dense_ffn": Family("dense_ffn", 2048, 1, 1, 8192, 6, (8, 2048)),
    # the large prefill batch's router and tokens (same seed) with I = 128
    # experts: profiles of the routing kernels within about 1 GB of device
    # memory
    "large_router": Family("large_router", 6144, 512, 12, 128, 5, (4096,), bias_std=1.0),
}

# tensor ids of the counter-based streams
TID_X, TID_ROUTER_W, TID_ROUTER_BIAS, TID_W13, TID_W2 = 1, 2, 3, 4, 5


def family(name: str) -> Family:
    try:
        return FAMILIES[name]
    except KeyError:
        raise KeyError(f"unknown workload family {name!r}; have {sorted(FAMILIES)}") from None


def workload_name(fam: Family, T: int) -> str:
    return f"{fam.name}_T{T}"


def parse_workload(name: str) -> tuple[Family, int]:
    """'olmoe_decode_T8' -> (family, 8)."""
    base, _, t = name.rpartition("_T")
    if not base or not t.isdigit():
        raise ValueError(f"workload name must look like <family>_T<tokens>, got {name!r}")
    return family(base), int(t)
