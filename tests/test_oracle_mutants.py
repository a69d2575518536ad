"""Plant plausible mistakes in a copy of the oracle's C source, build each
mutant on the CPU, and check that at least one pin fails for every mutant.
This shows the pins constrain the oracle, not just exercise it."""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    "scale_dropped": ("s *= scale;", ";"),
    "self_slot_excluded": ("const int64_t last = length + t;", "const int64_t last = length + t - 1;"),
    "one_future_slot": ("const int64_t last = length + t;", "const int64_t last = length + t + (length + t + 1 < M);"),
    "gqa_modulo_mapping": ("const int64_t kv = h / group;", "const int64_t kv = h % Hk;"),
    "no_max_subtraction": ("scratch[j] = exp(scratch[j] - m);", "scratch[j] = exp(scratch[j]);"),
    "query_row_fixed": ("at4(Hq, Q, D, b, h, t, d)", "at4(Hq, Q, D, b, h, 0, d)"),
    "lengths_not_advanced": ("out_lengths[b] = L + n;", "out_lengths[b] = L;"),
    "fp16_exponent_bias": ("e - 25", "e - 24"),
    "bf16_shift": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "non_prefix_accepted": ("if (mask_row[t]) f |= KVO_FLAG_MASK;", ";"),
    "softmax_epsilon": ("att_row[j] = scratch[j] / l;", "att_row[j] = scratch[j] / (l + 1e-9);"),
    # read-only re-attention
    "attend_self_slot_excluded": ("const int64_t last = K - S + t;", "const int64_t last = K - S + t - 1;"),
    "attend_slot_ignored": ("const int64_t slot = slot_ids ? slot_ids[b] : b;", "const int64_t slot = b;"),
    "attend_query_row_fixed": ("const int64_t row = cu_q[b] + t;", "const int64_t row = cu_q[b];"),
    "attend_s_gt_k_accepted": ("const int bad = S < 0 || S > K ||", "const int bad = S < 0 ||"),
    # gradients
    "bwd_softmax_not_centred": ("const double ds = a[j] * (g[j] - dot_ag);",
                                "const double ds = a[j] * g[j];"),
    "bwd_scale_dropped_in_dq": ("dq[d] += scale * ds * kd;", "dq[d] += ds * kd;"),
    "bwd_value_grad_from_ds": ("+= a[j] * dc;", "+= ds * dc;"),
    "bwd_overwritten_slot_keeps_grad": ("d_key_cache[at4(Hk, M, D, b, kv, j, d)] = 0.0;",
                                        "d_key_cache[at4(Hk, M, D, b, kv, j, d)] = gk;"),
    "bwd_new_row_offset": ("d_new_key[at4(Hk, Q, D, b, kv, j - L, d)] += scale * ds * qd;",
                           "d_new_key[at4(Hk, Q, D, b, kv, 0, d)] += scale * ds * qd;"),
}


def _fails_some_pin(o):
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            return pin.__name__
    return None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    c.write_text(mutated)
    lib = oracle.compile_library(str(c), str(tmp_path / f"lib{name}.so"))
    caught = _fails_some_pin(oracle.Oracle(lib))
    assert caught is not None, f"no pin catches mutant {name}"
