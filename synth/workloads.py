"""The five decode workloads of the CSA2 path, one chunked-prefill workload
and one encoder-side group (2 tokens per entry: a Full layer and five Reuse
layers), as sizes and seeds.

Each workload is seeded with 1000 + its index. Query token j of n_q sits at
absolute position t = N - n_q + j, where N counts the entries in the cache
after the step's new tokens have been appended. A prefill workload's n_q
tokens are one chunk of a prompt: each attends causally, with the exact
128-position window.
"""
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    mode: str           # "full" | "reuse" | "reindex" | "group"
    B: int              # sequences
    N: int              # context entries per sequence (after appending the step's tokens)
    n_q: int = 1        # query tokens per sequence
    layers: tuple = field(default=("full",))
    prefill: bool = False
    m: int = 1          # tokens per entry: 1 decoder layers, 2 encoder layers

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def queries(self) -> int:
        return self.B * self.n_q


WORKLOADS = {
    0: Workload(0, "full_b1_n32k", "full", B=1, N=32768),
    1: Workload(1, "reuse_b64_n64k", "reuse", B=64, N=65536, layers=("reuse",)),
    2: Workload(2, "reindex_b64_n128k", "reindex", B=64, N=131072, layers=("reindex",)),
    3: Workload(3, "full_b8_n1m", "full", B=8, N=1048576),
    4: Workload(4, "group_reindex_3reuse_b32_n256k_q6", "group", B=32, N=262144, n_q=6,
                layers=("reindex", "reuse", "reuse", "reuse")),
    5: Workload(5, "prefill_full_b1_n128k_c4096", "full", B=1, N=131072, n_q=4096, prefill=True),
    6: Workload(6, "encoder_full_5reuse_m2_b8_n1m", "group", B=8, N=1048576,
                layers=("full", "reuse", "reuse", "reuse", "reuse", "reuse"), m=2),
}

# Method constants (decoder CSA2 at m = 1).
LATENT_DIM = 512
IDX_HEADS = 32
IDX_DIM = 128
Q_HEADS = 64
TOPK = 512
POOL_BLOCKS = 2048
BLOCK = 8
WINDOW = 128
PAGE = 128
