"""The workloads the layer is measured and checked on.

Shapes follow the models the pages discuss: gpt-oss-20b (E=32, top-4,
hidden 2880, intermediate 2880; vLLM issue "moe_wna16_marlin_gemm applies wrong
per-row topk weights", Environment), gpt-oss-120b (E=128, hidden 2880; vLLM
issue "gpt-oss-120b MXFP4 + --enable-expert-parallel crashes") and
Nemotron-3-Nano (128 experts, top-6, hidden 2688, non-gated ReLU2, sigmoid+bias
routing; vLLM issue "... non-gated ReLU2 MoE (Nemotron-3-Nano)"). Nemotron's
intermediate size 1856 is not on the pages; it is the stated workload value.
"""
from dataclasses import dataclass, replace

FMT = {"nvfp4": 0, "mxfp4": 1, "int4": 2}
ACT = {"swigluoai": 0, "relu2": 1}
ROUTE = {"topk_softmax": 0, "sigmoid_bias": 1}


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    E: int
    k: int
    H: int
    I: int
    fmt: str
    act: str = "swigluoai"
    route: str = "topk_softmax"
    bias: bool = True
    zipf: float = 0.0          # logit[t, e] += -zipf * ln(e + 1)
    sel_bias_std: float = 0.0  # per-expert selection bias (sigmoid routing)
    w_std: float = 0.02
    x_std: float = 1.0
    bias_std: float = 0.01
    alpha: float = 1.702
    limit: float = 7.0
    workload: str = ""

    @property
    def gated(self) -> bool:
        return self.act == "swigluoai"

    @property
    def N1(self) -> int:
        return 2 * self.I if self.gated else self.I

    def with_T(self, T: int) -> "LayerConfig":
        return replace(self, T=T, name=f"{self.name.split('_t')[0]}_t{T}")


CONFIGS = {
    "c0": LayerConfig("c0", T=16, E=8, k=2, H=256, I=256, fmt="nvfp4",
                      workload="tiny MoE layer T16 E8 k2 H256 I256 NVFP4 swigluoai"),
    "c1": LayerConfig("c1", T=64, E=32, k=4, H=2880, I=2880, fmt="nvfp4",
                      workload="gpt-oss-20b-shaped decode layer T64 E32 k4 H2880 I2880 NVFP4 W4A16"),
    "c2": LayerConfig("c2", T=4096, E=32, k=4, H=2880, I=2880, fmt="int4", zipf=1.1,
                      workload="gpt-oss-20b-shaped prefill T4096 E32 k4 H2880 I2880 GPTQ-INT4 g64, Zipf(1.1) routing"),
    "c3_t1": LayerConfig("c3_t1", T=1, E=128, k=4, H=2880, I=2880, fmt="mxfp4",
                         workload="gpt-oss-120b-shaped layer T1 E128 k4 H2880 I2880 MXFP4"),
    "c3_t32": LayerConfig("c3_t32", T=32, E=128, k=4, H=2880, I=2880, fmt="mxfp4",
                          workload="gpt-oss-120b-shaped layer T32 E128 k4 H2880 I2880 MXFP4"),
    "c3_t8192": LayerConfig("c3_t8192", T=8192, E=128, k=4, H=2880, I=2880, fmt="mxfp4",
                            workload="gpt-oss-120b-shaped layer T8192 E128 k4 H2880 I2880 MXFP4"),
    "c4": LayerConfig("c4", T=2048, E=128, k=6, H=2688, I=1856, fmt="nvfp4", act="relu2",
                      route="sigmoid_bias", bias=False, sel_bias_std=0.1,
                      workload="Nemotron-3-Nano-shaped layer T2048 E128 k6 H2688 I1856 NVFP4 ReLU2"),
}


def get_config(key: str, **overrides) -> LayerConfig:
    cfg = CONFIGS[key]
    return replace(cfg, **overrides) if overrides else cfg
