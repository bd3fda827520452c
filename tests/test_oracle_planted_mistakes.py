"""Planted mistakes: every pin of the oracle must turn red under a plausible error.

Each case below copies the oracle's C++ source, makes one edit a reader could plausibly
make when writing it from the pages (a dropped term, a wrong sign, axis or operand, an
off-by-one), builds the copy with the oracle's own flags, loads it in place of the real
oracle, and runs the pins named for the case: every one of them has to fail.  A control
build of the unedited copy passes every pin named here, so the failures come from the
edits and not from the harness.  The edits are made on the CPU, in a temporary copy;
the committed oracle is never changed.
"""
import os
import shutil
import subprocess
from dataclasses import dataclass

import pytest

import oracle

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "gdn_oracle.cpp")


@dataclass(frozen=True)
class Pin:
    module: str
    test: str
    args: tuple = ()        # (name, value) pairs; "FD_CASES[i]" reads the module, a tuple
                            # value is passed as a list

    def run(self):
        mod = __import__(self.module)
        kw = {}
        for name, value in self.args:
            if isinstance(value, str) and value.startswith("FD_CASES["):
                value = mod.FD_CASES[int(value[len("FD_CASES["):-1])]
            elif isinstance(value, tuple):
                value = list(value)
            kw[name] = value
        getattr(mod, self.test)(**kw)

    def __str__(self):
        return "%s::%s%s" % (self.module, self.test, dict(self.args) if self.args else "")


@dataclass(frozen=True)
class Mistake:
    name: str
    old: str                # text of the oracle that the edit replaces
    new: str
    pins: tuple             # every one must fail on the edited oracle
    count: int = 1          # occurrences of `old` in the source
    nth: int = 0            # which occurrence is edited


P = "test_oracle_pins"
FD = Pin(P, "test_backward_matches_central_differences", (("case", "FD_CASES[1]"),))
FD_MULTI = Pin(P, "test_backward_matches_central_differences", (("case", "FD_CASES[3]"),))
T1 = Pin(P, "test_t1_closed_form_forward_and_backward")
B0G1 = Pin(P, "test_beta0_gate1_leaves_state_untouched")
B0 = Pin(P, "test_beta0_decays_state_by_softplus_gate")
SCALE = Pin(P, "test_query_key_scale_invariance")
SHARED = Pin(P, "test_shared_key_head_equals_explicit_repeat")
MODULO = Pin(P, "test_modulo_head_map_equals_consecutive_map_on_permuted_heads")
N = "test_oracle_neighbours"
CONV_FD = Pin(N, "test_conv_gradients_match_central_differences", (("K", 4), ("cu", (0, 5, 9))))
DELAY = Pin(N, "test_conv_oldest_tap_is_a_delay_line_reset_at_sequence_starts")
NORM_FD = Pin(N, "test_norm_gradients_match_central_differences",
              (("H", 1), ("D", 16), ("eps", 1e-2)))
CONST = Pin(N, "test_norm_of_a_constant_row", (("D", 4),))
C = "test_oracle_context"
AFFINE = Pin(C, "test_final_state_is_affine_in_the_start_state",
             (("Hk", 2), ("Hv", 4), ("head_map", 0)))
DECAY = Pin(C, "test_no_write_strength_leaves_pure_decay")
K_ = "test_oracle_kda"
KDA_EQ = Pin(K_, "test_equal_channel_gates_reduce_to_the_scalar_gate", (("Hk", 1), ("Hv", 2)))
KDA_FD = Pin(K_, "test_gradients_match_central_differences")
KDA_UNTOUCHED = Pin(K_, "test_untouched_channels_only_decay")

KDA_DECAY_THEN_READ = (
    "  for (int i = 0; i < d.Dk; ++i)\n"
    "    for (int j = 0; j < d.Dv; ++j) S[(int64_t)i * d.Dv + j] *= g[i];\n"
    "  for (int j = 0; j < d.Dv; ++j) kv[j] = 0.0;\n"
    "  for (int i = 0; i < d.Dk; ++i)\n"
    "    for (int j = 0; j < d.Dv; ++j) kv[j] += S[(int64_t)i * d.Dv + j] * khat[i];\n")
KDA_READ_THEN_DECAY = (
    "  for (int j = 0; j < d.Dv; ++j) kv[j] = 0.0;\n"
    "  for (int i = 0; i < d.Dk; ++i)\n"
    "    for (int j = 0; j < d.Dv; ++j) kv[j] += S[(int64_t)i * d.Dv + j] * khat[i];\n"
    "  for (int i = 0; i < d.Dk; ++i)\n"
    "    for (int j = 0; j < d.Dv; ++j) S[(int64_t)i * d.Dv + j] *= g[i];\n")

MISTAKES = [
    # --- the recurrence, forward ---
    Mistake("retrieval_not_decayed",
            "delta[j] = G.b * (v[j] - G.g * kv[j]);", "delta[j] = G.b * (v[j] - kv[j]);",
            (FD, T1)),
    Mistake("l2_eps_1e-3",
            "const double n = std::sqrt(ss + 1e-6);", "const double n = std::sqrt(ss + 1e-3);",
            (T1, B0G1, SCALE)),
    Mistake("key_in_place_of_query_in_output",
            "orow[j] += Sh[(int64_t)i * d.Dv + j] * qh[i];",
            "orow[j] += Sh[(int64_t)i * d.Dv + j] * kh_[i];", (FD, T1, B0G1)),
    Mistake("beta_without_sigmoid",
            "G.b = sigmoid(in.beta_raw[t * in.beta_ld + h]);",
            "G.b = in.beta_raw[t * in.beta_ld + h];", (FD, T1)),
    Mistake("softplus_without_log_term",
            "return std::max(x, 0.0) + std::log1p(std::exp(-std::fabs(x)));",
            "return std::max(x, 0.0);", (FD, T1, B0)),
    Mistake("dt_bias_dropped",
            "G.x = in.alpha[t * in.alpha_ld + h] + in.dt_bias[h];",
            "G.x = in.alpha[t * in.alpha_ld + h];", (FD, B0)),
    Mistake("modulo_map_by_default",
            "return head_map ? kh + hh * Hk : kh * r + hh;", "return kh + hh * Hk;",
            (SHARED, MODULO)),
    # --- the recurrence, backward ---
    Mistake("retrieval_adjoint_into_dk_dropped",
            "dkh[i] += S_prev[(int64_t)i * d.Dv + j] * dkv[j];", "dkh[i] += 0.0 * dkv[j];",
            (FD, T1)),
    Mistake("state_adjoint_not_decayed",
            "for (size_t e = 0; e < SZ; ++e) dSh[e] *= G.g;",
            "for (size_t e = 0; e < SZ; ++e) dSh[e] *= 1.0;", (FD, T1)),
    Mistake("d_a_log_without_log_gate",
            "pa[(size_t)n * d.Hv + h] += dl * G.l;", "pa[(size_t)n * d.Hv + h] += dl;",
            (FD, T1)),
    Mistake("d_beta_raw_without_sigmoid_slope",
            "dbeta_raw[t * dbeta_ld + h] = db * G.b * (1.0 - G.b);",
            "dbeta_raw[t * dbeta_ld + h] = db;", (FD, T1)),
    Mistake("l2_backward_without_projection",
            "dq_acc[i] += (dqh[i] - qh[i] * dot_q) / nq;", "dq_acc[i] += dqh[i] / nq;",
            (FD, T1), count=2, nth=0),
    Mistake("recompute_segment_one_token_short",
            "tb = std::min<int64_t>(ta + seg, t1);", "tb = std::min<int64_t>(ta + seg - 1, t1);",
            (FD, FD_MULTI)),
    # --- conv1d + SiLU and gated RMSNorm ---
    Mistake("conv_taps_reversed",
            "const int64_t src = t - (K - 1 - j);\n    if (src >= t_start)",
            "const int64_t src = t - j;\n    if (src >= t_start)", (CONV_FD, DELAY)),
    Mistake("conv_buffer_carried_across_sequences",
            "if (src >= t_start) s +=", "if (src >= 0) s +=", (CONV_FD, DELAY)),
    Mistake("silu_slope_as_sigmoid_slope",
            "return s * (1.0 + x * (1.0 - s));", "return s * (1.0 - s);", (CONV_FD, NORM_FD)),
    Mistake("rms_of_the_sum",
            "const double rms = std::sqrt(ss / D + eps);", "const double rms = std::sqrt(ss + eps);",
            (CONST, NORM_FD), count=2, nth=0),
    Mistake("eps_outside_the_root",
            "const double rms = std::sqrt(ss / D + eps);",
            "const double rms = std::sqrt(ss / D) + eps;", (CONST, NORM_FD), count=2, nth=0),
    # --- state map (context parallelism) ---
    Mistake("state_map_without_beta",
            "(P[(int64_t)i * d.Dk + j] - G.b * kh_[i] * w[j])",
            "(P[(int64_t)i * d.Dk + j] - kh_[i] * w[j])", (AFFINE,)),
    Mistake("state_map_without_decay",
            "= G.g * (P[(int64_t)i * d.Dk + j] -", "= (P[(int64_t)i * d.Dk + j] -",
            (AFFINE, DECAY)),
    Mistake("state_map_transposed_product",
            "w[j] += kh_[i] * P[(int64_t)i * d.Dk + j];",
            "w[j] += kh_[i] * P[(int64_t)j * d.Dk + i];", (AFFINE,)),
    # --- KDA ---
    Mistake("kda_retrieval_before_the_decay", KDA_DECAY_THEN_READ, KDA_READ_THEN_DECAY,
            (KDA_EQ, KDA_FD)),
    # g holds Dk gates; the pins below run Dk = 4 >= Dv = 3, so g[j] stays in bounds
    Mistake("kda_gate_on_value_channels",
            "for (int j = 0; j < d.Dv; ++j) S[(int64_t)i * d.Dv + j] *= g[i];",
            "for (int j = 0; j < d.Dv; ++j) S[(int64_t)i * d.Dv + j] *= g[j];",
            (KDA_FD, KDA_UNTOUCHED)),
    Mistake("kda_last_channel_dropped_from_dg",
            "dg[i] = acc;", "dg[i] = i + 1 < d.Dk ? acc : 0.0;", (KDA_FD,)),
    Mistake("kda_d_b_alpha_from_dl",
            "pb[((size_t)n * d.Hv + h) * d.Dk + c] += dx;",
            "pb[((size_t)n * d.Hv + h) * d.Dk + c] += dl;", (KDA_FD, KDA_EQ)),
]


def _edit(src: str, m: Mistake) -> str:
    assert src.count(m.old) == m.count, (m.name, src.count(m.old))
    at = -1
    for _ in range(m.nth + 1):
        at = src.index(m.old, at + 1)
    return src[:at] + m.new + src[at + len(m.old):]


@pytest.fixture(scope="module")
def builds(tmp_path_factory):
    """Every edited copy and the control, compiled in parallel with the oracle's flags."""
    if shutil.which("g++") is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("planted")
    with open(SRC) as f:
        src = f.read()
    jobs = {}
    for name, text in [("control", src)] + [(m.name, _edit(src, m)) for m in MISTAKES]:
        cpp, so = d / (name + ".cpp"), d / (name + ".so")
        cpp.write_text(text)
        jobs[name] = (str(so), subprocess.Popen(["g++"] + oracle.compile_flags() +
                                                [str(cpp), "-o", str(so)],
                                                stderr=subprocess.PIPE))
    out = {}
    for name, (so, proc) in jobs.items():
        _, err = proc.communicate()
        assert proc.returncode == 0, (name, err.decode()[-2000:])
        out[name] = so
    return out


def _failures(lib_path, pins, monkeypatch):
    failed = []
    with monkeypatch.context() as mp:
        mp.setattr(oracle, "_lib", oracle.open_library(lib_path))
        for pin in pins:
            try:
                pin.run()
            except AssertionError:
                failed.append(pin)
    return failed


def test_unedited_copy_passes_every_named_pin(builds, monkeypatch):
    pins = list(dict.fromkeys(p for m in MISTAKES for p in m.pins))
    assert _failures(builds["control"], pins, monkeypatch) == []


@pytest.mark.parametrize("m", MISTAKES, ids=lambda m: m.name)
def test_planted_mistake_fails_its_pins(m, builds, monkeypatch):
    failed = _failures(builds[m.name], m.pins, monkeypatch)
    missed = [str(p) for p in m.pins if p not in failed]
    assert not missed, "pins that stayed green: %s" % missed
