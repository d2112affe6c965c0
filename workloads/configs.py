"""The five synthetic attention workloads: shapes, seeds and budget targets.

These are plain facts about the inputs (sizes, seeds, distributions).  No step
of the sparse-attention method is computed here.

Shapes follow the attention layers of the models the S-HPLB pages evaluate on
(Llama-3.1-8B, Qwen2.5-7B, Qwen2.5-72B; S-HPLB page, "Risultati Sperimentali"
and the Chinese page, section 4) at up to 128K tokens of context.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    number: int
    name: str
    mode: str                      # "prefill" or "decode"
    seq_len: int                   # S (prefill) or cache length L (decode)
    block: int                     # B, tokens per block
    num_q_heads: int               # Hq
    num_kv_heads: int              # Hkv
    head_dim: int                  # d
    batch: int                     # sequences
    q_scale_lo: float              # s_h ~ log-uniform in [lo, hi]
    q_scale_hi: float
    target_density: float          # mean fraction of causal blocks (prefill)
    demand_source: str             # "coverage", "lognormal" or "decode"
    lognormal_sigma: float = 0.0
    heavy_keys: int = 0            # planted heavy-key positions per KV head
    streaming_fraction: float = 0.0
    window_tokens: int = 0         # decode: streaming window
    budget_tokens: int = 0         # decode: retrieval budget
    calib_len_cap: int = 8192      # calibration draw length cap

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def calib_seed(self) -> int:
        """Seed of the calibration draw (distinct from every workload seed)."""
        return 2000 + self.number

    @property
    def nb(self) -> int:
        return self.seq_len // self.block

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def calib_len(self) -> int:
        return min(self.seq_len, self.calib_len_cap)


WORKLOADS = {
    1: Workload(1, "tiny_prefill_4k", "prefill", 4096, 64, 8, 2, 64, 1,
                0.5, 3.0, 0.25, "coverage"),
    2: Workload(2, "llama31_8b_prefill_32k", "prefill", 32768, 128, 32, 8, 128, 1,
                0.5, 4.0, 0.10, "coverage"),
    3: Workload(3, "llama31_8b_prefill_128k", "prefill", 131072, 128, 32, 8, 128, 1,
                0.5, 4.0, 0.06, "coverage"),
    4: Workload(4, "qwen25_72b_prefill_128k", "prefill", 131072, 128, 64, 8, 128, 1,
                0.5, 4.0, 0.06, "lognormal", lognormal_sigma=1.0, heavy_keys=4),
    5: Workload(5, "qwen25_7b_decode_64k", "decode", 65536, 32, 28, 4, 128, 16,
                0.5, 4.0, 0.0, "decode", streaming_fraction=0.4,
                window_tokens=2048, budget_tokens=2048),
}


def workload(number: int) -> Workload:
    return WORKLOADS[number]


def scaled(w: Workload, seq_len: int, num_q_heads: int | None = None,
           num_kv_heads: int | None = None, batch: int | None = None) -> Workload:
    """The same recipe at another size (used for small test cases)."""
    from dataclasses import replace
    return replace(w, seq_len=seq_len,
                   num_q_heads=num_q_heads or w.num_q_heads,
                   num_kv_heads=num_kv_heads or w.num_kv_heads,
                   batch=batch or w.batch)
