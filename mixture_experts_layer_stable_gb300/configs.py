"""Named workloads of the single-GPU MoE layer.

Shapes follow the layer the Mixture-of-Kittens pages benchmark (hidden 7168,
expert intermediate 2048 -- leiphone "MoK..." section 02, minibatch paragraph)
plus a tiny parity case and a balanced mid-size case.
"""

from dataclasses import dataclass, field, asdict


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int            # tokens
    d: int            # hidden size
    f: int            # expert intermediate size
    E: int            # experts
    k: int            # top-k
    logit_std: float  # router logits ~ N(0, logit_std) (+ Zipf bias when zipf > 0)
    zipf: float = 0.0
    prec: str = "bf16"          # "bf16" or "mxfp8"
    passes: str = "fwd"         # "fwd" or "fwd+bwd"
    minibatch_rows: tuple = field(default_factory=tuple)

    @property
    def R(self) -> int:
        return self.T * self.k

    def as_dict(self):
        return asdict(self)


CONFIGS = {
    "tiny": LayerConfig("tiny", T=64, d=128, f=64, E=8, k=2, logit_std=1.0,
                        passes="fwd+bwd"),
    "balanced": LayerConfig("balanced", T=2048, d=2048, f=768, E=64, k=8,
                            logit_std=0.1, minibatch_rows=(1024,)),
    "kimi_zipf": LayerConfig("kimi_zipf", T=4096, d=7168, f=2048, E=256, k=8,
                             logit_std=1.0, zipf=1.2,
                             minibatch_rows=(512, 1024, 2368, 2560, 4096)),
    "kimi_mxfp8": LayerConfig("kimi_mxfp8", T=4096, d=7168, f=2048, E=256, k=8,
                              logit_std=0.1, prec="mxfp8"),
    "kimi_bwd": LayerConfig("kimi_bwd", T=2048, d=7168, f=2048, E=256, k=8,
                            logit_std=1.0, zipf=1.2, passes="fwd+bwd"),
    # one GPU's share of the pages' expert-parallel run (64-way: 4 experts of
    # the Kimi-like shape and about 4,096 rows each per GPU), reproduced on one
    # GPU as k = 1 over 4 experts: the compute-bound end of the layer
    "local_slice": LayerConfig("local_slice", T=16384, d=7168, f=2048, E=4, k=1,
                               logit_std=0.1),
    # the Kimi-like expert shape at a size whose profiler captures stay within
    # a few GB of device memory (2.8 GB of weights, 22 of 32 experts with
    # fewer than 128 rows, as most experts of the Zipf-routed layer)
    "kimi_small": LayerConfig("kimi_small", T=512, d=7168, f=2048, E=32, k=8,
                              logit_std=1.0, zipf=1.2),
}
