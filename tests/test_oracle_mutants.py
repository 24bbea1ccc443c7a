"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (the pins are strong enough to notice a dropped term,
a wrong sign, a wrong index or a swapped operand).  CPU only."""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests.oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, original text, planted mistake); every original occurs exactly once
MUTANTS = [
    ("scale_dropped", "srow[j] = scale * dot;", "srow[j] = dot;"),
    ("exp_sign_flipped", "exp(srow[j] - m);", "exp(m - srow[j]);"),
    ("not_normalised", "srow[j] /= l;", "srow[j] /= 1.0;"),
    ("causal_masks_diagonal", "if (causal && j > pos) {", "if (causal && j >= pos) {"),
    ("causal_mask_transposed", "if (causal && j > pos) {", "if (causal && j < pos) {"),
    ("causal_chunk_top_left", "const long pos = i + (Nk - Nq);", "const long pos = i;"),
    ("causal_chunk_offset_sign", "const long pos = i + (Nk - Nq);",
     "const long pos = i + (Nq - Nk);"),
    ("lse_without_max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("lse_base2", "*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    ("scores_use_v", "is_bf16) *\n                   load_elem(k, kvbase",
     "is_bf16) *\n                   load_elem(v, kvbase"),
    ("bwd_dq_uses_v", "dqi[c] += scale * ds * load_elem(k,", "dqi[c] += scale * ds * load_elem(v,"),
    ("output_uses_k", "o_row[c] += srow[j] * load_elem(v,", "o_row[c] += srow[j] * load_elem(k,"),
    ("online_no_rescale", "l * exp(m - m_new)) + s;", "l) + s;"),
    ("merge_sign_flipped", "exp(m1 - m);", "exp(m - m1);"),
    ("blocked_no_o_rescale", "acc[r * d + c] = alpha * acc[r * d + c] + pv;",
     "acc[r * d + c] = acc[r * d + c] + pv;"),
    ("blocked_skips_diagonal_block", "if (causal && j0 > i0 + br - 1 + off)",
     "if (causal && j0 > i0 + off)"),
    ("blocked_chunk_stops_early", "if (causal && j0 > i0 + br - 1 + off)",
     "if (causal && j0 > i0 + br - 1)"),
    ("blocked_chunk_top_left", "if (!(causal && j > i + off)) {", "if (!(causal && j > i)) {"),
    ("bf16_widening_shift", "(uint32_t)bits << 16;", "(uint32_t)bits << 15;"),
    ("bwd_D_dropped", "const double ds = p * (dprow[j] - D);", "const double ds = p * dprow[j];"),
    ("bwd_dq_no_scale", "dqi[c] += scale * ds * kjc;", "dqi[c] += ds * kjc;"),
    ("bwd_dk_uses_k", "+= scale * ds * qic;", "+= scale * ds * kjc;"),
    ("bwd_dv_uses_ds", "+= p * doic;", "+= ds * doic;"),
    ("bwd_dp_uses_k", "is_bf16) *\n                  load_elem(v, kvbase",
     "is_bf16) *\n                  load_elem(k, kvbase"),
    ("bwd_rows_D_dropped", "prow[j] * (dprow[j] - Di);", "prow[j] * dprow[j];"),
    ("bwd_keys_lse_sign", "exp(scale * s - lse[i]);", "exp(scale * s + lse[i]);"),
    ("bwd_keys_top_left", "if (causal && j > i + (Nk - Nq))\n                    continue;",
     "if (causal && j > i)\n                    continue;"),
    ("bwd_keys_dv_uses_q", "dvj[c] += p * load_elem(dout,", "dvj[c] += p * load_elem(q,"),
    ("mx_scale_bias", "return ldexp(1.0, (int)code - 127);", "return ldexp(1.0, (int)code - 128);"),
    ("mx_block_index", "e8m0_value(scales[r * nb + c / block])", "e8m0_value(scales[r * nb + c % nb])"),
    ("mx_scale_dropped", "e8m0_value(scales[r * nb + c / block]) * e4m3_value",
     "1.0 * e4m3_value"),
    ("mx_nan_code", "if (code == 0xFF)\n        return NAN;", "if (code == 0xFE)\n        return NAN;"),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path_c = tmp_path / f"{name}.c"
    path_c.write_text(src.replace(old, new))
    path_so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-ffp-contract=off",
                    str(path_c), "-o", str(path_so), "-lm"], check=True)
    return oracle._declare(ctypes.CDLL(str(path_so)))


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new):
    lib = _build_mutant(tmp_path, name, old, new)
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(oracle)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin noticed the planted mistake {name!r}"
