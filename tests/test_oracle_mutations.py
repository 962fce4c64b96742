"""The pins must catch plausible mistakes.

Each case plants one mistake in a private copy of the oracle's C source,
builds it with gcc into a temporary library, swaps it in, and checks that
at least one pin of ``test_oracle_pins`` fails against it.  Runs on the CPU
only; the real oracle is left untouched.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "swa_oracle.c")

MUTATIONS = {
    # the window holds W+1 keys instead of W
    "window_off_by_one": ("int64_t a = p - window + 1;", "int64_t a = p - window;"),
    # draft rows see later draft rows
    "no_causality": ("*hi = p < seq_len - 1 ? p : seq_len - 1;", "*hi = seq_len - 1;"),
    # query head h reads KV head h mod Hkv instead of floor(h / G)
    "gqa_modulo": ("const int64_t g = h / G;", "const int64_t g = h % J->Hkv;"),
    # max dropped from the log-sum-exp
    "lse_drops_max": ("J->lse[row] = m + log(z);", "J->lse[row] = log(z);"),
    # merge rescales with the wrong sign
    "merge_sign": ("const double w = exp(mk - M);", "const double w = exp(M - mk);"),
    # q and k dims transposed in the score (reads k at the wrong stride)
    "score_operand": ("dot += qr[d] * kr[d];", "dot += qr[d] * kr[(d * 7) % D];"),
    # argmax ties go to the last column instead of the first
    "argmax_last_tie": ("if (row[j] > best) {", "if (row[j] >= best) {"),
    # the acceptance compares a draft with the next row's token
    "accept_wrong_row": ("while (n < q_len - 1 && argmax[b * q_len + n] == draft[b * (q_len - 1) + n]) ++n;",
                         "while (n < q_len - 1 && argmax[b * q_len + n + 1] == draft[b * (q_len - 1) + n]) ++n;"),
    # the append writes up to the cache end instead of stopping at seq_len
    "append_no_seq_len_clip": ("const int64_t end = seq_lens[b] < L ? seq_lens[b] : L;",
                               "const int64_t end = L;"),
    # the new rows read as [B, Hkv, q_len, D] instead of [B, q_len, Hkv, D]
    "append_rows_layout": ("const double *src = rows + ((b * q_len + i) * Hkv + h) * D;",
                           "const double *src = rows + ((b * Hkv + h) * q_len + i) * D;"),
    # row i lands one position late
    "append_row_offset": ("const int64_t pos = q_pos[b] + i;", "const int64_t pos = q_pos[b] + i + 1;"),
    # the window holds W-1 keys (the query's own key dropped at the far edge)
    "window_short": ("int64_t a = p - window + 1;", "int64_t a = p - window + 2;"),
    # rows past the cached context see the key at seq_len
    "seq_len_clip_inclusive": ("*hi = p < seq_len - 1 ? p : seq_len - 1;",
                               "*hi = p < seq_len ? p : seq_len;"),
    # the score misses the scale
    "scale_dropped": ("s[j - lo] = J->scale * dot;", "s[j - lo] = dot;"),
    # softmax weights not divided by their sum
    "weights_unnormalised": ("const double w = s[j - lo] / z; /* = exp(s_j - lse) */",
                             "const double w = s[j - lo];"),
    # lse reported in log2 units
    "lse_log2": ("J->lse[row] = m + log(z);", "J->lse[row] = (m + log(z)) / log(2.0);"),
    # a partial's key range includes its end key (chunks overlap by one)
    "partial_range_inclusive": ("if (hi > J->c_hi[b] - 1) hi = J->c_hi[b] - 1;",
                                "if (hi > J->c_hi[b]) hi = J->c_hi[b];"),
    # the merge's denominator forgets the partials' rescaling
    "merge_lambda_unscaled": ("Lam += l[k * rows + r] * w;", "Lam += l[k * rows + r];"),
    # the accepted count includes the bonus token
    "accept_counts_bonus": ("accepted[b] = n;", "accepted[b] = n + 1;"),
    # the keep set's relabelling skipped
    "accept_keep_ignored": ("argmax[b * q_len + i] = keep ? keep[jbest] : jbest;",
                            "argmax[b * q_len + i] = jbest;"),
}

PIN_CHECKS = [
    lambda: [pins.test_hand_worked_examples(c) for c in pins._load_golden()],
    lambda: pins.test_brute_force_tiny(8),
    lambda: pins.test_brute_force_gqa_batch_ragged(),
    lambda: pins.test_brute_force_prefill_block(),
    lambda: pins.test_full_window_is_causal_attention(64, 2, 1, 40, 8),
    lambda: [pins.test_split_merge_identity(n) for n in (2, 3)],
    lambda: pins.test_zero_keys_closed_form(),
    lambda: [pins.test_accept_hand_worked_examples(c) for c in pins._load_accept_golden()],
    lambda: pins.test_accept_matches_numpy_argmax_and_prefix_count(),
    lambda: [pins.test_append_hand_worked_examples(c) for c in pins._load_append_golden()],
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                    str(lib), str(mutated), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle._bind(str(lib)))
    failures = 0
    for check in PIN_CHECKS:
        try:
            check()
        except (AssertionError, ValueError):
            failures += 1
    assert failures > 0, f"no pin caught mutation {name}"
