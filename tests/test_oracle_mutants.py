"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, points the oracle module at the mutant
and runs a quick set of pins; at least one pin must fail.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import oracle as _oracle_mod

import test_oracle_pins as pins
import test_oracle_ring_step as steps
import test_oracle_ffn as ffn_pins

SRC = os.path.join(os.path.dirname(pins.__file__), "..", "oracle", "ring_attn_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("static int n_visible(const problem_t *P, int i) { return P->causal ? i + 1 : P->L; }",
                          "static int n_visible(const problem_t *P, int i) { return P->causal ? i + 2 - (i + 1 >= P->L) : P->L; }"),
    "gqa_head_map": ("const int g = h / (P->Hq / P->Hkv);\n  const double *qi = q_row(P, b, h, i);\n  const int n",
                     "const int g = h % P->Hkv;\n  const double *qi = q_row(P, b, h, i);\n  const int n"),
    "lse_drops_max": ("const double lse = m + log(sum);", "const double lse = log(sum) + (m > 0 ? 0 : m);"),
    "dq_missing_scale": ("(dpij - D);\n    const double *kj = k_row(P, b, g, j);\n    for (int c = 0; c < P->d; ++c) dq[c] += P->scale * dsij * kj[c];",
                         "(dpij - D);\n    const double *kj = k_row(P, b, g, j);\n    for (int c = 0; c < P->d; ++c) dq[c] += dsij * kj[c];"),
    "ds_missing_D": ("const double dsij = pij * (dpij - D);", "const double dsij = pij * dpij;"),
    "dk_wrong_operand": ("(dpij - D[base + i]);\n      for (int c = 0; c < P->d; ++c) {\n        dv[c] += pij * doi[c];\n        dk[c] += P->scale * dsij * qi[c];",
                         "(dpij - D[base + i]);\n      for (int c = 0; c < P->d; ++c) {\n        dv[c] += pij * doi[c];\n        dk[c] += P->scale * dsij * doi[c];"),
    "dv_uses_ds": ("(dpij - D[base + i]);\n      for (int c = 0; c < P->d; ++c) {\n        dv[c] += pij * doi[c];\n        dk[c] += P->scale * dsij * qi[c];",
                   "(dpij - D[base + i]);\n      for (int c = 0; c < P->d; ++c) {\n        dv[c] += dsij * doi[c];\n        dk[c] += P->scale * dsij * qi[c];"),
    "merge_wrong_sign": ("const double a = exp(*lse - merged), w = exp(lse_s - merged);",
                         "const double a = exp(*lse - merged), w = exp(merged - lse_s);"),
    "fold_wrong_pair": ("return sub < N ? sub : 2 * N - 1 - sub;", "return sub < N ? sub : sub - N;"),
    "merge_weights_swapped": ("for (int c = 0; c < d; ++c) oa[c] = wa * oa[c] + wb * ob[c];",
                              "for (int c = 0; c < d; ++c) oa[c] = wb * oa[c] + wa * ob[c];"),
    "step_wrong_source": ("if (!ring_block(P, t->n_chunks, b, h, i, t->src, s, o_s, &lse_s, t->schedule)) {",
                          "if (!ring_block(P, t->n_chunks, b, h, i, t->rank, s, o_s, &lse_s, t->schedule)) {"),
    "stripes_as_blocks": ("if (schedule == SCHED_STRIPED) return p % N;",
                          "if (schedule == SCHED_STRIPED) return p / (L / N);"),
    "dfa_helper_wrong_keys": ("    *q_chunk = N - t + w;\n    *kv_chunk = w;",
                              "    *q_chunk = N - t + w;\n    *kv_chunk = (w - t + N) % N;"),
    "dfa_middle_launch_doubled": ("  if (t < N - t) {", "  if (t <= N - t) {"),
    "dfa_last_launch_dropped": ("for (int launch = 0; launch <= N / 2; ++launch)",
                                "for (int launch = 0; launch < N / 2; ++launch)"),
    "block_bwd_mask_dropped": ("owner_rank(P->L, t->n_chunks, P->causal, t->schedule, j) == t->src && (!P->causal || j <= i);",
                               "owner_rank(P->L, t->n_chunks, P->causal, t->schedule, j) == t->src;"),
    "block_bwd_dv_uses_ds": ("t->D[base + i]);\n      for (int c = 0; c < P->d; ++c) {\n        dv[c] += pij * doi[c];",
                             "t->D[base + i]);\n      for (int c = 0; c < P->d; ++c) {\n        dv[c] += dsij * doi[c];"),
    "contiguous_as_fold": ("if (!causal || schedule != SCHED_FOLD) return p / (L / N);",
                           "if (!causal) return p / (L / N);"),
    "ffn_residual_dropped": ("y[c] = x[c] + acc[c];", "y[c] = acc[c];"),
    "ffn_gelu_wrong_scale": ("return 0.5 * erfc(-x / sqrt(2.0));", "return 0.5 * erfc(-x / 2.0);"),
    "ffn_cdf_wrong_sign": ("return 0.5 * erfc(-x / sqrt(2.0));", "return 0.5 * erfc(x / sqrt(2.0));"),
    "ffn_gelu_grad_missing_term": ("return Phi + x * phi;", "return Phi;"),
    "ffn_dx_residual_dropped": ("for (int c = 0; c < f->D; ++c) dx[c] = dy[c];", "for (int c = 0; c < f->D; ++c) dx[c] = 0.0;"),
    "ffn_dw2_wrong_operand": ("for (int c = 0; c < f->D; ++c) dw2[c] += hm * dy[c];",
                              "for (int c = 0; c < f->D; ++c) dw2[c] += hm * x[c];"),
    "ffn_dw1_uses_h": ("f->dw1[(size_t)c * f->F + j] += x[c] * dam;", "f->dw1[(size_t)c * f->F + j] += x[c] * hm;"),
    "ffn_db1_sums_h": ("db1 += dam;", "db1 += hm;"),
    "ffn_da_uses_gelu": ("da[j] = dh * gelu_grad(a);", "da[j] = dh * gelu(a);"),
    "ffn_dx_transposed_w1": ("dx[c] += da[j] * w[(size_t)c * f->F + j];", "dx[c] += da[j] * w[(size_t)j * f->D + c];"),
    "rows_stats_start_late": ("lo[bh] = causal ? kmin : 0;", "lo[bh] = causal ? kmin + 1 : 0;"),
    "rows_dq_wrong_row": ("dq_row(P, b, h, t->rows[ri], lse, D, t->dq + ((size_t)bh * t->n_rows + ri) * P->d);",
                          "dq_row(P, b, h, t->rows[ri], lse, D, t->dq + ((size_t)bh * t->n_rows + (t->n_rows - 1 - ri)) * P->d);"),
    "transposed_score": ("s[j] = P->scale * dot(qi, k_row(P, b, g, j), P->d);\n    if (s[j] > m) m = s[j];\n  }\n  double sum",
                         "s[j] = P->scale * dot(q_row(P, b, h, j), k_row(P, b, g, i), P->d);\n    if (s[j] > m) m = s[j];\n  }\n  double sum"),
}


def _quick_pins():
    """Run a fast subset of the pins; return the names of those that fail."""
    checks = [
        ("sdpa_fwd", lambda: [pins.test_fwd_matches_torch_sdpa(s, c) for s in pins.SHAPES[:2] for c in (False, True)]),
        ("sdpa_bwd", lambda: [pins.test_bwd_matches_torch_autograd(s, c) for s in pins.SHAPES[:2] for c in (False, True)]),
        ("rows_sum", lambda: [pins.test_softmax_rows_sum_to_one(c) for c in (False, True)]),
        ("ring", lambda: [pins.test_ring_form_invariant_in_chunk_count(48, c) for c in (False, True)]),
        ("row0", pins.test_causal_row_zero_closed_form),
        ("gqa", lambda: [pins.test_gqa_equals_repeated_mha(c) for c in (False, True)]),
        ("fold", lambda: [pins.test_fold_gives_every_rank_equal_causal_work(n) for n in (2, 4)]),
        ("hand", lambda: [pins.test_hand_worked_example(m) for m in ("enc", "cau")]),
        ("steps", lambda: [steps.test_steps_merged_in_ring_order_equal_plain(48, 3, c, st)
                           for c in (False, True) for st in (False, True)]),
        ("merge", steps.test_merge_weights_are_a_sigmoid_of_the_lse_gap),
        ("stripes", lambda: steps.test_striped_step_with_zero_queries_closed_form(3)),
        ("dfa", lambda: [steps.test_contiguous_causal_ring_forms_equal_plain(L, N, sc)
                         for L, N in ((48, 3), (64, 4), (60, 5)) for sc in ("contiguous", "dfa")]),
        ("contiguous", lambda: steps.test_contiguous_step_with_zero_queries_closed_form(3)),
        ("block_bwd", lambda: [steps.test_backward_blocks_sum_to_the_plain_backward(sc, True)
                               for sc in ("fold", "contiguous")]),
        ("ffn", lambda: [ffn_pins.test_ffn_matches_torch(7, 16, 64), ffn_pins.test_gelu_values()]),
        ("ffn_bwd", lambda: ffn_pins.test_ffn_backward_matches_torch_autograd(5, 8, 24)),
        ("rows", lambda: [pins.test_row_sampled_routines_agree_with_full(c) for c in (False, True)]),
    ]
    failed = []
    for name, fn in checks:
        try:
            with np.errstate(all="ignore"):
                fn()
        except Exception:  # any failure or error counts as a caught mutant
            failed.append(name)
    return failed


def test_unmutated_source_passes_quick_pins():
    assert _quick_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(mut),
                           "-lm", "-lpthread"])
    prev = _oracle_mod._swap_library(str(so))
    try:
        failed = _quick_pins()
    finally:
        _oracle_mod._restore_library(prev)
    assert failed, f"mutant {name} passed every pin"
    # the real oracle is back in place
    assert oracle.owner_rank(8, 2, True, 7) == 0
