"""The measured workloads use the pages' lengths (CPU only)."""
import os

from long_causal_gqa_gb300.inputs import WORKLOADS, HEADLINE

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "failing_sequence_lengths.txt")


def _failing_lengths():
    out = []
    with open(GOLDEN) as fh:
        for line in fh:
            if line.startswith("#") or "|" not in line:
                continue
            cells = [c.strip() for c in line.split("|")]
            if cells[2] == "fail":
                out.append(int(cells[3]))
    return out


def test_golden_table_parses():
    assert sorted(_failing_lengths()) == [8184, 8199, 8510, 10231]


def test_varlen_workload_packs_the_failing_lengths():
    assert sorted(WORKLOADS["varlen4"].seqlens) == sorted(_failing_lengths())


def test_headline_is_the_issue_title_length():
    assert WORKLOADS[HEADLINE].seqlens == (max(_failing_lengths()),)
    w = WORKLOADS[HEADLINE]
    assert (w.n_q_heads, w.n_kv_heads, w.head_dim) == (64, 8, 128)
    # metric FLOPs: 2 * S^2 * Hq * D
    assert abs(w.metric_flops() - 2 * 10231 ** 2 * 64 * 128) < 1


def test_under_limit_and_outlier_workloads():
    assert WORKLOADS["s7700"].seqlens == (7700,)
    assert WORKLOADS["s32768_outlier"].n_outlier == 4
    assert WORKLOADS["s512"].total_tokens == 512
