"""Plant plausible mistakes in a copy of the oracle and check the pins catch
each one.  The mistakes are planted in the oracle source, on the CPU only."""
import os
import shutil
import subprocess

import pytest

import oracle_pins
from oracle import build as obuild

# (name, original text, planted text): a dropped term, a wrong sign or index,
# a transposed operand, an off-by-one mask, a wrong normaliser.
MUTANTS = [
    ("drop_scale", "s[j] = scale * dot;", "s[j] = dot;"),
    ("k_is_v", "qi[d] * K[(size_t)j * D + d]", "qi[d] * V[(size_t)j * D + d]"),
    ("causal_off_by_one", "&& j > i) return 0;", "&& j >= i) return 0;"),
    ("causal_flipped", "&& j > i) return 0;", "&& j < i) return 0;"),
    ("padding_off_by_one", "if (j >= len) return 0;", "if (j > len) return 0;"),
    ("no_max_shift", "s[j] = exp(s[j] - M);", "s[j] = exp(s[j]);"),
    ("no_normalise", "double w = s[j] / Z;", "double w = s[j];"),
    ("min_not_max", "if (!any || s[j] > M) M = s[j];", "if (!any || s[j] < M) M = s[j];"),
    ("unbiased_var", "var /= N;", "var /= (N - 1);"),
    ("eps_outside", "1.0 / sqrt(var + eps)", "1.0 / (sqrt(var) + eps)"),
    ("gamma_beta_swapped", "* rstd * gamma[c] + beta[c]", "* rstd * beta[c] + gamma[c]"),
    ("head_split_transposed",
     "x[((size_t)b * Lq + i) * (size_t)H * D + (size_t)h * D + d];",
     "x[((size_t)b * Lq + i) * (size_t)H * D + (size_t)d * H + h];"),
    ("pv_uses_k", "o[d] += w * V[(size_t)j * D + d];", "o[d] += w * K[(size_t)j * D + d];"),
    ("length_of_batch0", "int len = kv_lengths[b];", "int len = kv_lengths[0];"),
    ("rows_api_head_index", "size_t bh = (size_t)b * H + (size_t)h;\n        attend_row",
     "size_t bh = (size_t)h * B + (size_t)b;\n        attend_row"),
    ("residual_dropped", "out[e] = x[e] + out[e];", "out[e] = out[e];"),
    ("residual_doubled", "out[e] = x[e] + out[e];", "out[e] = x[e] + x[e] + out[e];"),
    ("residual_rows_wrong_head",
     "(size_t)i) * (size_t)H * D + (size_t)h * D;\n        for (int d = 0;",
     "(size_t)i) * (size_t)H * D;\n        for (int d = 0;"),
    ("bwd_drop_row_term", "double dS = p[j] * (dP[j] - c);", "double dS = p[j] * dP[j];"),
    ("bwd_row_term_sign", "c += p[j] * dP[j];", "c -= p[j] * dP[j];"),
    ("bwd_dP_uses_k", "dP[j] += gi[d] * V[", "dP[j] += gi[d] * K["),
    ("bwd_dq_uses_v", "dQ[(size_t)i * D + d] += scale * dS * K[", "dQ[(size_t)i * D + d] += scale * dS * V["),
    ("bwd_dk_unscaled", "dK[(size_t)j * D + d] += scale * dS * qi[d];",
     "dK[(size_t)j * D + d] += dS * qi[d];"),
    ("bwd_dv_uses_dS", "dV[(size_t)j * D + d] += p[j] * gi[d];", "dV[(size_t)j * D + d] += dS * gi[d];"),
    ("lse_drops_max", "lse[bh * Lq + (size_t)i] = M + log(Z);", "lse[bh * Lq + (size_t)i] = log(Z);"),
]


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


def test_unmutated_oracle_passes_all_pins():
    assert oracle_pins.run_all() == []


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(workdir, name, orig, planted):
    src = open(obuild.SRC).read()
    assert src.count(orig) == 1, "mutation anchor not unique: %s" % name
    path = os.path.join(str(workdir), name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(orig, planted))
    lib = os.path.join(str(workdir), "lib%s.so" % name)
    obuild.build(force=True, src=path, out=lib)
    fails = oracle_pins.run_all(path=lib)
    assert fails, "mutant %s survived every pin" % name
