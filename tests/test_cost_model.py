"""The FLOP model bench.py reports: 2 * H * D per (query, record).

FlashMemory-DeepSeek-V4 gives per-decode-token whole-model FLOPs at 1M context
("Highlights" and "Per-decode-token FLOPs (whole model)"): 118.9 GFLOP with the
native indexer scoring the whole history, 35.4 GFLOP when Level 2 scores only
the resident set, and 26.6 GFLOP of constant work in both. The scoring parts are
therefore 92.3 and 8.8 GFLOP. "Two-level recall algorithm" fixes the counts the
model needs: Level 2 runs every step over all 21 c4 layers; Level 1 (the Memory
Indexer, H = 128 in its training command) scores the full history at 3 target
layers once every 64 steps; and "Quick start" gives KMAX = 384 pages of 64
records at 1M. With 2^20 tokens compressed 4:1 (262144 records) the model gives
90.2 and 8.86 GFLOP; the 2% gap on the first is the page's "1M" being slightly
more than 2^20 tokens (a 1.07M-token history reproduces it exactly), and the
second lands within 1%. A model that dropped the factor 2, used D = 64, or
counted H = 128 for Level 2 misses both figures by far more.
"""
import numpy as np
import pytest

import bench
from sparse_attention_kv_e4m3_gb300 import synth

WHOLE_FULL, WHOLE_RESIDENT, CONSTANT = 118.9, 35.4, 26.6
LAYERS_L2, LAYERS_L1, HEADS_L1, EVERY = 21, 3, 128, 64
RECORDS_1M = (1 << 20) // 4
KMAX_1M = 384


def test_full_history_scoring_reproduces_the_baseline_indexer_part():
    model = bench.indexer_gflop(LAYERS_L2, RECORDS_1M)
    page = WHOLE_FULL - CONSTANT  # 92.3
    assert abs(model - 90.19) < 0.01
    assert abs(model - page) / page < 0.03
    # the history length at which the model gives the page's figure exactly: ~1.07M tokens
    tokens = page * 1e9 / (LAYERS_L2 * 2 * 64 * 128) * 4
    assert 1.05e6 < tokens < 1.10e6


def test_resident_scoring_and_level1_reproduce_the_flashmemory_part():
    level2 = bench.indexer_gflop(LAYERS_L2, KMAX_1M * 64)
    level1 = bench.indexer_gflop(LAYERS_L1, RECORDS_1M, heads=HEADS_L1) / EVERY
    page = WHOLE_RESIDENT - CONSTANT  # 8.8
    assert abs(level2 - 8.456) < 0.001 and abs(level1 - 0.403) < 0.001
    assert abs(level2 + level1 - page) / page < 0.01
    # the whole-model ratio the page quotes (0.30x)
    assert abs((CONSTANT + level2 + level1) / (CONSTANT + bench.indexer_gflop(LAYERS_L2, RECORDS_1M)) - 0.30) < 0.01


@pytest.mark.parametrize("wrong", ["no_factor_2", "d64", "h128"])
def test_plausible_mistakes_miss_the_pages_figures(wrong):
    f = {"no_factor_2": lambda L, n: L * n * 64 * 128 / 1e9,
         "d64": lambda L, n: L * n * 2 * 64 * 64 / 1e9,
         "h128": lambda L, n: L * n * 2 * 128 * 128 / 1e9}[wrong]
    assert abs(f(LAYERS_L2, RECORDS_1M) - (WHOLE_FULL - CONSTANT)) / (WHOLE_FULL - CONSTANT) > 0.3


def test_bench_counts_flops_per_visible_record():
    # ragged rows, one empty, a resident subset: the count follows the visible records only
    w = synth.make_workload("flops", num_q=4, history=[700, 0, 64 * 9 + 5, 3000], seed=3)
    vis = w.visible_counts()
    assert bench.algorithmic_flops(w) == 2 * 64 * 128 * int(vis.sum())
    r = synth.make_workload("flops_res", num_q=2, history=[64 * 40, 64 * 30], resident_pages=7, seed=4)
    assert bench.algorithmic_flops(r) == 2 * 64 * 128 * int(r.visible_counts().sum())
    assert int(r.visible_counts().sum()) <= 2 * 7 * 64
    # config 4's count: the causal mask's visible records summed over its 4096 queries
    p = synth.config("prefill_chunk")
    assert bench.algorithmic_flops(p) == 2 * 64 * 128 * int(np.asarray(p.visible_counts()).sum())
