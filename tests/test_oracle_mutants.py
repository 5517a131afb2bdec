"""Planted mistakes in the oracle (on the CPU) must be caught by its pins.

Each case rewrites one line of an oracle function (a flipped comparison, a
dropped term, a wrong index), installs the rewritten function in the oracle
module for the duration of the test, and checks that at least one of the
pins in ``test_oracle_pins.py`` then fails.
"""
import inspect
import textwrap

import pytest

import oracle
import oracle.ring_attention as ra
import test_oracle_pins as pins
import test_oracle_window_variant as wv
import test_oracle_usp as usp
import test_oracle_decode as dec


def _mutant(func, old, new):
    src = textwrap.dedent(inspect.getsource(func))
    assert src.count(old) >= 1, (func.__name__, old)
    src = src.replace(old, new)
    ns = {}
    exec(compile(src, f"<mutant {func.__name__}>", "exec"), ra.__dict__, ns)
    return ns[func.__name__]


CASES = [
    # (function, original text, planted text, pins that should catch it)
    ("partial_attention", "kh = h // G", "kh = h % Hkv",
     [pins.test_cp1_equals_library_causal_sdpa]),
    ("_vis", "(kp[None, :] <= qp[:, None])", "(kp[None, :] < qp[:, None])",
     [lambda: pins.test_forward_matches_brute_force(None),
      pins.test_worked_example_load_balance]),
    ("_vis", "< window", "<= window",
     [lambda: wv.test_window_forward_matches_brute_force(3, None)]),
    ("_vis", "(kd[None, :] == qd[:, None])", "(kd[None, :] <= qd[:, None])",
     [lambda: pins.test_forward_matches_brute_force([0, 5, 6, 13, 20])]),
    ("select_variant", "q_msg < kv_msg", "q_msg <= kv_msg",
     [wv.test_select_variant_crossover_is_the_message_size_tie]),
    ("select_variant", "2 * (n_new + n_cached) * n_kv_heads", "2 * n_cached * n_kv_heads",
     [wv.test_select_variant_follows_the_pages,
      wv.test_select_variant_crossover_is_the_message_size_tie]),
    ("partial_attention", "mx_safe + np.log(l_safe)", "np.log(l_safe)",
     [lambda: pins.test_forward_matches_brute_force(None)]),
    ("partial_attention", "np.exp(s - mx_safe[:, None])", "np.exp(s)",
     [lambda: pins.test_forward_matches_brute_force(None)]),
    ("doc_index", 'side="right"', 'side="left"',
     [lambda: pins.test_forward_matches_brute_force([0, 5, 6, 13, 20])]),
    ("rank_chunks", "[r, 2 * R - 1 - r]", "[r, R + r]",
     [pins.test_worked_example_load_balance]),
    ("rank_chunks", "for c in (d, 2 * D - 1 - d)", "for c in (d, D + d)",
     [usp.test_usp_figure_pairs_of_devices,
      lambda: usp.test_usp_ranks_balanced_and_increasing(2, 2)]),
    ("head_split", "x[:, u * hs:(u + 1) * hs]", "x[:, u:u + hs]",
     [usp.test_head_split_moves_heads_not_tokens]),
    ("decode", "[T - 1], np.arange(r * n, (r + 1) * n)", "[n - 1], np.arange(r * n, (r + 1) * n)",
     [lambda: dec.test_decode_is_the_last_row_of_causal_attention(2)]),
    ("decode", "v[b, r * n:(r + 1) * n]", "v[b, 0:n]",
     [lambda: dec.test_decode_is_the_last_row_of_causal_attention(4)]),
    ("ring_schedule", "row.append((r, other))", "row.append((r, r))",
     [lambda: pins.test_ring_equals_monolithic("pass_kv", "zigzag", False)]),
    ("lse_merge", "np.exp(lses - LSE_safe[None])", "np.exp(lses - M_safe[None])",
     [lambda: pins.test_ring_equals_monolithic("pass_q", "zigzag", False)]),
    ("plan_positions", """            if cache is not None:
                kv_pos[r].append(cache[r])
            kv_pos[r].append(new[r])""",
     """            kv_pos[r].append(new[r])
            if cache is not None:
                kv_pos[r].append(cache[r])""",
     [pins.test_partial_prefill_plan]),
    ("plan_positions", "offset=b * L + P, a2a=a2a)", "offset=b * int(seq_len) + P, a2a=a2a)",
     [pins.test_batch_positions_partition_and_balance]),
    ("round_bf16", "np.rint(a0 / spacing)", "np.floor(a0 / spacing)",
     [pins.test_round_bf16_hand_values, pins.test_round_bf16_matches_torch_conversion]),
    ("round_bf16", "np.maximum(e, -125)", "np.maximum(e, -200)",
     [pins.test_round_bf16_hand_values, pins.test_round_bf16_matches_torch_conversion]),
    ("round_bf16", "np.ldexp(1.0, e - 8)", "np.ldexp(1.0, e - 7)",
     [pins.test_round_bf16_hand_values, pins.test_round_bf16_matches_torch_conversion]),
    ("ring_forward", 'round_bf16(o_t) if partial_dtype == "bf16" else o_t', "o_t",
     [pins.test_ring_forward_bf16_partials_pass_q]),
    ("work_list", "items.sort(key=lambda it: -(it[4] - it[3]))",
     "items.sort(key=lambda it: it[4] - it[3])",
     [pins.test_work_list_closed_forms]),
    ("work_list", "lo, hi = int(nz[0]), int(nz[-1]) + 1", "lo, hi = int(nz[0]), int(nz[-1])",
     [pins.test_work_list_closed_forms]),
    ("_pair_backward", "ds = p * (dp - D[h, r0:r1][:, None])", "ds = p * dp",
     [lambda: pins.test_backward_finite_differences(None)]),
    ("_pair_backward", "dq[r0:r1, h, :] += scale * (ds @ kk)",
     "dq[r0:r1, h, :] += (ds @ kk)",
     [pins.test_backward_equals_library_autograd]),
    ("_pair_backward", "dv[ksel, kh, :] += p.T @ dout[r0:r1, h, :]",
     "dv[ksel, kh, :] += p.T @ dout[r0:r1, kh, :]",
     [pins.test_backward_equals_library_autograd]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}:{c[2]}" for c in CASES])
def test_planted_mistake_is_caught(case, monkeypatch):
    name, old, new, checks = case
    fn = _mutant(getattr(ra, name), old, new)
    monkeypatch.setattr(ra, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)
    caught = 0
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught > 0, f"planted mistake in {name} was not caught"
