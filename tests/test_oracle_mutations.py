"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pin suite (test_oracle_pins.py) fails for every one of them.

Each mutation is a small textual edit of ``oracle/moe_oracle.c`` compiled into
a scratch copy of the oracle package; the real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "nibble_order": ("(i % 2 == 0) ? (byte & 0xF) : (byte >> 4)", "(i % 2 == 1) ? (byte & 0xF) : (byte >> 4)"),
    "exponent_bias_128": ("e8m0 - 127", "e8m0 - 128"),
    "sign_bit": ("(code & 8) ? -m : m", "(code & 4) ? -m : m"),
    "magnitude_order": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 6.0, 4.0}"),
    "block_of_16": ("sr[i / 32]", "sr[i / 16 % (cols/32)]"),
    "tie_to_higher_index": ("return a->idx < b->idx ? -1 : (a->idx > b->idx ? 1 : 0);",
                            "return a->idx < b->idx ? 1 : (a->idx > b->idx ? -1 : 0);"),
    "no_renormalisation": ("for (int j = 0; j < k; ++j)\n            denom += exp",
                           "for (int j = 0; j < E; ++j)\n            denom += exp"),
    "unstable_permutation": ("for (int64_t s = 0; s < n; ++s) {\n        int32_t p",
                             "for (int64_t s = n - 1; s >= 0; --s) {\n        int32_t p"),
    "gate_up_swapped": ("h[n] = g / (1.0 + exp(-g)) * u;", "h[n] = u / (1.0 + exp(-u)) * g;"),
    "shared_dropped": ("acc += y[(t * nsel + k + s) * H + m];", "acc += 0.0;"),
    "silu_sign": ("g / (1.0 + exp(-g))", "g / (1.0 + exp(g))"),
    "slice_dropped": ("for (int j = 0; j < ns; ++j) {", "for (int j = 0; j < (ns > 1 ? ns - 1 : ns); ++j) {"),
    "down_transposed": ("const float *wd = Wd + (int64_t)m * ld_d;\n        for (int n = 0; n < I; ++n)\n"
                        "            acc += h[n] * (double)wd[n];",
                        "for (int n = 0; n < I; ++n)\n            acc += h[n] * (double)Wd[(int64_t)n * ld_d + m % ld_d];"),
    "weights_reversed": ("acc += w[t * k + j] * y", "acc += w[t * k + (k - 1 - j)] * y"),
    "empty_slot_weight_read": ("if (ids[t * k + j] != -1)\n                        acc +=", "if (1)\n                        acc +="),
    "empty_slot_placed_last": ("int32_t p = ids[s] == -1 ? -1 : next[ids[s]]++;",
                               "int32_t p = ids[s] == -1 ? (int32_t)(n - 1) : next[ids[s]]++;"),
    "sigmoid_bias_in_weights": ("w[t * k + j] = scale * score[s[j].idx] / denom;",
                                "w[t * k + j] = scale * s[j].v / denom;"),
    "sigmoid_bias_ignored": ("s[e].v = score[e] + (bias ? (double)bias[e] : 0.0);", "s[e].v = score[e];"),
    "sigmoid_sign": ("score[e] = 1.0 / (1.0 + exp(-(double)logits[t * E + e]));",
                     "score[e] = 1.0 / (1.0 + exp((double)logits[t * E + e]));"),
    "i4_nibble_order": ("(i & 1) ? (byte >> 4) : (byte & 0xF)", "(i & 1) ? (byte & 0xF) : (byte >> 4)"),
    "i4_zero_sign": ("(double)(q - z)", "(double)(z - q)"),
    "i4_zero_ignored": ("(double)(q - z)", "(double)(q - 8)"),
    "i4_group_of_16": ("r * ng + i / 32", "r * ng + (i / 16) % ng"),
    "i4_default_zero_0": ("zeros ? zeros[grp] : 8", "zeros ? zeros[grp] : 0"),
    "i4_zero_16_accepted": ("|| z > 15)", "|| z > 16)"),
    "fp16_exponent_bias_16": ("ex - 25", "ex - 26"),
    "fp16_subnormal_flushed": ("v = ldexp((double)fr, -24);", "v = 0.0;"),
    "fp16_implicit_bit_dropped": ("ldexp((double)(1024 + fr), ex - 25)", "ldexp((double)fr, ex - 25)"),
    "sigmoid_normalised_over_all": ("for (int j = 0; j < k; ++j)\n            denom += score[s[j].idx];",
                                    "for (int e = 0; e < E; ++e)\n            denom += score[e];"),
}


@pytest.fixture(scope="module")
def scratch():
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(d, "tests"),
                    ignore=shutil.ignore_patterns("__pycache__", "test_oracle_mutations.py", "test_*gpu*", "test_zz*"))
    os.makedirs(os.path.join(d, "mxfp4_routed_expert_router_gb300"))
    for f in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "mxfp4_routed_expert_router_gb300", f),
                    os.path.join(d, "mxfp4_routed_expert_router_gb300", f))
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(scratch, name):
    old, new = MUTATIONS[name]
    src = open(os.path.join(ROOT, "oracle", "moe_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    odir = os.path.join(scratch, "oracle")
    shutil.rmtree(odir, ignore_errors=True)
    os.makedirs(odir)
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), odir)
    with open(os.path.join(odir, "moe_oracle.c"), "w") as f:
        f.write(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-q", "-x", "-p", "no:warnings",
                        "-p", "no:cacheprovider"], cwd=scratch, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1 and "failed" in r.stdout, f"mutation {name} survived:\n{r.stdout[-2000:]}"
