"""The pins must catch a wrong oracle.  Each case plants one plausible
mistake in a copy of the oracle (a dropped term, a wrong sign, offset or
index, a swapped operand, another rounding or tie rule), builds or loads that
copy on the CPU, and runs the oracle pins against it: at least one pin has to
fail.  The oracle itself is never modified."""
import ctypes
import importlib.util
import os
import subprocess
import sys

import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_policy as ppins
from conftest import read_golden

# (name, exact text in oracle/moe_oracle.c, replacement)
C_MUTANTS = [
    ("q4 offset 7", "return orc_code(blk, i) - 8;", "return orc_code(blk, i) - 7;"),
    ("q4 nibbles swapped", "return i < 16 ? (qs[i] & 15) : (qs[i - 16] >> 4);",
     "return i < 16 ? (qs[i] >> 4) : (qs[i - 16] & 15);"),
    ("silu on up", "double h = g * u / (1.0 + exp(-g));", "double h = g * u / (1.0 + exp(-u));"),
    ("top-k tie to the higher index", "if (best < 0 || l[e] > l[best]) best = e;",
     "if (best < 0 || l[e] >= l[best]) best = e;"),
    ("round half away from zero", "float r = rintf(xb[i] / dd);", "float r = roundf(xb[i] / dd);"),
    ("activation scale dropped", "double term = orc_h2d(orc_block_scale(blk)) * orc_h2d(da[b]) * (double)s;",
     "double term = orc_h2d(orc_block_scale(blk)) * (double)s;"),
    ("routing weight dropped", "for (int i = 0; i < H; ++i) yt[i] += w[a] * o[i];",
     "for (int i = 0; i < H; ++i) yt[i] += o[i];"),
    ("scale over 128", "float d32 = amax / 127.0f;", "float d32 = amax / 128.0f;"),
    ("q8 codes unsigned", "if (fmt == 1) return (int)(int8_t)blk[2 + i];", "if (fmt == 1) return (int)blk[2 + i];"),
    ("q5 fifth-bit index", "const int hi = (qh[i / 8] >> (i % 8)) & 1;", "const int hi = (qh[i % 4] >> (i / 4)) & 1;"),
    ("q5 offset 15", "if (fmt == 2) return orc_code5(blk, i) - 16;", "if (fmt == 2) return orc_code5(blk, i) - 15;"),
    ("q4k scale from the wrong nibble", "*sc = (b[j + 4] & 15) | ((b[j - 4] >> 6) << 4);",
     "*sc = (b[j + 4] >> 4) | ((b[j - 4] >> 6) << 4);"),
    ("q4k min added in the dot", "acc += da_b * (p1 - p2);", "acc += da_b * (p1 + p2);"),
    ("q4k min added in dequant", "out[(size_t)s * 256 + i] = d * sc * (double)orc_k4_code(sb, i) - dmin * m;",
     "out[(size_t)s * 256 + i] = d * sc * (double)orc_k4_code(sb, i) + dmin * m;"),
    ("q4k sub-block halves swapped", "return r < 32 ? (qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4);",
     "return r < 32 ? (qs[32 * c + r] >> 4) : (qs[32 * c + r - 32] & 15);"),
    ("binary16 truncation", "double r = nearbyint(a / quantum); /* default rounding: ties to even */",
     "double r = floor(a / quantum);"),
    ("softmax over all logits", "if (renorm) {", "if (!renorm) {"),
    ("q6k high pair index", "const int hi = (qh[32 * n + l] >> (2 * m)) & 3;",
     "const int hi = (qh[i % 64] >> (2 * (i / 64))) & 3;"),
    ("q6k low nibble byte", "const uint8_t lb = ql[64 * n + 32 * (m & 1) + l];",
     "const uint8_t lb = ql[64 * n + 32 * (m >> 1) + l];"),
    ("q5k fifth bit index", "return lo | (((qh[l] >> j) & 1) << 4);", "return lo | (((qh[j] >> l) & 1) << 4);"),
    ("q5k code bytes offset", "const uint8_t *qh = sb + 16, *qs = sb + 48;", "const uint8_t *qh = sb + 16, *qs = sb + 44;"),
    ("q2k quarter shift", "return (qs[32 * n + t] >> (2 * m)) & 3;", "return (qs[32 * n + t] >> m) & 3;"),
    ("q2k min from the low nibble", "*m = sb[j] >> 4;", "*m = sb[j] & 15;"),
    ("q2k min added in the dot", "acc += da_s * (sq - mq);", "acc += da_s * (sq + mq);"),
    ("q3k high bit sense", "return ((hm[t] >> (4 * n + m)) & 1) ? low : low - 4;",
     "return ((hm[t] >> (4 * n + m)) & 1) ? low - 4 : low;"),
    ("q3k scale high pair", "const int high2 = (b[8 + j % 4] >> (2 * (j / 4))) & 3;",
     "const int high2 = (b[8 + j / 4] >> (2 * (j % 4))) & 3;"),
    ("q6k offset 31", "t += (int32_t)(orc_k6_code(sb, e) - 32) * (int32_t)qa[e];",
     "t += (int32_t)(orc_k6_code(sb, e) - 31) * (int32_t)qa[e];"),
]

# oracle pins that take no fixture, and those that take the golden reader
C_PINS = [pins.test_h2d_all_bit_patterns_vs_numpy, pins.test_f2h_vs_numpy_random_and_ties,
          pins.test_topk_signed_zero_tie_goes_to_lower_index, pins.test_topk_brute_force_subsets,
          pins.test_topk_weights_closed_forms, pins.test_quantizer_brute_force_and_scale,
          pins.test_quantizer_exact_ties_round_half_even, pins.test_block_dot_brute_force,
          pins.test_dequant_vs_independent, pins.test_row_dot_vs_dense_fp64, pins.test_layer_vs_dense_fp64_brute_force,
          pins.test_q8_block_dot_brute_force_and_extremes, pins.test_q8_dequant_vs_independent,
          pins.test_q8_row_dot_vs_dense_fp64, pins.test_q8_layer_vs_dense_fp64_brute_force,
          pins.test_quantizer_zero_and_tiny_blocks, pins.test_q5_block_dot_brute_force_every_code,
          pins.test_q5_dequant_and_layer_vs_dense_fp64, pins.test_q4k_brute_force_vs_independent_decode,
          pins.test_q4k_layer_vs_dense_fp64, pins.test_shared_expert_layer_vs_dense_fp64,
          pins.test_q6k_brute_force_vs_independent_decode, pins.test_q6k_layer_vs_dense_fp64,
          pins.test_q5k_brute_force_vs_independent_decode, pins.test_q5k_layer_vs_dense_fp64,
          pins.test_q2k_brute_force_vs_independent_decode, pins.test_q2k_layer_vs_dense_fp64,
          pins.test_q3k_brute_force_vs_independent_decode, pins.test_q3k_layer_vs_dense_fp64]
C_GOLDEN_PINS = [pins.test_h2d_golden, pins.test_block_dot_golden, pins.test_q8_block_dot_golden,
                 pins.test_q5_block_dot_golden, pins.test_q4k_golden, pins.test_q6k_golden, pins.test_q5k_golden,
                 pins.test_q2k_golden, pins.test_q3k_golden]


def _failing_pins(run):
    failed = []
    for f in C_PINS:
        try:
            run(f, ())
        except Exception:  # an assertion, or a mutant that breaks a call
            failed.append(f.__name__)
    for f in C_GOLDEN_PINS:
        try:
            run(f, (read_golden,))
        except Exception:
            failed.append(f.__name__)
    return failed


def _build_mutant(old, new, tmp):
    with open(oracle._SRC) as f:
        src = f.read()
    assert src.count(old) == 1, old
    path = os.path.join(tmp, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    out = os.path.join(tmp, "libmutant.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", path, "-o",
                    out, "-lm"], check=True)
    return oracle.configure(ctypes.CDLL(out))


@pytest.mark.parametrize("name,old,new", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_numeric_oracle_mutant_fails_a_pin(name, old, new, tmp_path):
    mutant = _build_mutant(old, new, str(tmp_path))
    saved = oracle.lib()
    oracle._lib = mutant
    try:
        failed = _failing_pins(lambda f, a: f(*a))
    finally:
        oracle._lib = saved
    assert failed, f"no pin catches the mutant '{name}'"


def test_unmutated_oracle_passes_every_pin():
    assert _failing_pins(lambda f, a: f(*a)) == []


# (name, exact text in oracle/policy.py, replacement)
P_MUTANTS = [
    ("window boundary <=", "if not (ls >= 0 and self.clock - ls < self.window):",
     "if not (ls >= 0 and self.clock - ls <= self.window):"),
    ("admit on the first sighting", "if not (ls >= 0 and self.clock - ls < self.window):",
     "if not (ls >= -1 and self.clock - ls < self.window):"),
    ("stamp tie to the higher slot",
     "if t.stamp[s] < self.clock and (best is None or t.stamp[s] < t.stamp[best]):",
     "if t.stamp[s] < self.clock and (best is None or t.stamp[s] <= t.stamp[best]):"),
    ("shared-pool tie to the higher slot",
     "if self.g_stamp[g] < self.clock and (best is None or self.g_stamp[g] < self.g_stamp[best]):",
     "if self.g_stamp[g] < self.clock and (best is None or self.g_stamp[g] <= self.g_stamp[best]):"),
    ("placed expert keeps its sighting", "                t.last_seen[e] = -1\n            swaps += 1",
     "                pass\n            swaps += 1"),
    ("preheat ranks by fewest uses", "return (-c, self.t[tid].rank[e], tid)", "return (c, self.t[tid].rank[e], tid)"),
    ("hits not stamped", "                        t.stamp[s] = self.clock\n", "                        pass\n"),
    ("shared-pool hits not stamped", "                        self.g_stamp[s] = self.clock\n",
     "                        pass\n"),
    ("admissions while slots are lent", "        if self.n_lent == 0:\n            self._admit(misses)",
     "        if True:\n            self._admit(misses)"),
    ("lent tail off by one", "return list(range(G - n, G))", "return list(range(G - n - 1, G - 1))"),
]

P_PINS = [ppins.test_hand_traced_max_swaps, ppins.test_invariants_and_brute_force_misses_long_run,
          ppins.test_admission_needs_second_sighting_within_window, ppins.test_hand_traced_preheat_per_tensor,
          ppins.test_global_pool_of_one_tensor_is_the_per_tensor_policy,
          ppins.test_global_pool_invariants_and_misses_long_run]
P_GOLDEN_PINS = [ppins.test_hand_traced_sequence, ppins.test_hand_traced_borrow_return,
                 ppins.test_hand_traced_global_pool]


def _load_policy_mutant(old, new, tmp):
    with open(os.path.join(os.path.dirname(oracle.__file__), "policy.py")) as f:
        src = f.read()
    assert src.count(old) == 1, old
    path = os.path.join(tmp, "policy_mutant.py")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("policy_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules["policy_mutant"] = mod
    spec.loader.exec_module(mod)
    return mod.PolicyOracle


@pytest.mark.parametrize("name,old,new", P_MUTANTS, ids=[m[0] for m in P_MUTANTS])
def test_policy_oracle_mutant_fails_a_pin(name, old, new, tmp_path, monkeypatch):
    monkeypatch.setattr(ppins, "PolicyOracle", _load_policy_mutant(old, new, str(tmp_path)))
    failed = []
    for f in P_PINS:
        try:
            f()
        except Exception:
            failed.append(f.__name__)
    for f in P_GOLDEN_PINS:
        try:
            f(read_golden)
        except Exception:
            failed.append(f.__name__)
    assert failed, f"no pin catches the policy mutant '{name}'"
