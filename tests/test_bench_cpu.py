"""Host-side arithmetic of bench.py's reports, on hand-countable cases (no GPU)."""
import numpy as np

import bench
from workloads import inputs


def _case(ids, n_kv=2):
    ids = np.asarray(ids, dtype=np.int32)
    nq = ids.shape[0]
    H = 16 * n_kv
    return inputs.AttnCase(qa=np.zeros((nq, H, 128), np.uint16), kc=np.zeros((n_kv, 256, 128), np.uint16),
                           vc=None, ids=ids, n_tokens=np.full(nq, 256, np.int32), scale=1.0)


def test_attention_bytes_count_every_selection_once_per_kv_head():
    c = _case([[0, 1, -1], [1, 2, 3]], n_kv=2)        # 5 selections, 2 KV heads
    per_selection = 2 * 64 * 128 * 2                   # K and V of one block, bf16
    qa_out_lse = 2 * 32 * (128 * 2 + 128 * 4 + 4)      # q in, out and lse, per query and head
    want = 5 * 2 * per_selection + qa_out_lse + 4 * c.ids.size + 4 * 2
    assert bench.attention_bytes(c) == want


def test_attention_unique_bytes_count_each_distinct_block_once():
    c = _case([[0, 1, -1], [1, 2, 3]], n_kv=2)        # distinct blocks 0, 1, 2, 3
    assert bench.attention_unique_bytes(c) == 4 * 2 * 32768


def test_job_figures_scale_with_the_ranks():
    assert bench.job_us_per_call(0.024, 1) == 24.0
    assert abs(bench.job_us_per_call(0.024, 4) - 6.0) < 1e-12


def test_parity_report_on_a_tiny_case_counts_every_query():
    """The bench's parity block from the oracle's own fp32-rounded scores: rule (a)
    identical, rule (b) error at fp32 rounding, rule (c) every query exact."""
    import oracle
    case = inputs.tiny_case()
    ref = oracle.block_scores(case.q, case.w, case.kblk, case.n_blocks, case.dtype)
    gpu_scores = ref.astype(np.float32)
    ids = oracle.select_f32(gpu_scores, case.n_blocks, case.k)
    rep = bench.parity_report(case, gpu_scores, ids, ids, "chained")
    assert rep["rule_a"] == {"identical_queries": case.nq, "pass": True}
    assert rep["rule_b"]["pass"] and rep["rule_b"]["max_normalised_error"] < 1e-6
    assert rep["rule_c"]["pass"] and rep["rule_c"]["exact"] == case.nq and rep["rule_c"]["failed"] == 0


def test_event_times_are_averaged_not_snapped():
    # four calls timed at the ~2 us steps of the event timer (ms in, us out): the mean, not the median
    assert abs(bench.us_mean([0.002048, 0.002048, 0.004096, 0.002048]) - 2.56) < 1e-9
