"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one of them (mutation testing, CPU only)."""
import os
import tempfile

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

# (name, original text, mutated text)
MUTANTS = [
    ("renorm dropped", "    if (norm) {\n        double s = 0.0;", "    if (0) {\n        double s = 0.0;"),
    ("top-k picks smallest", "probs[e] > probs[best]", "probs[e] < probs[best]"),
    ("ties go to higher index", "probs[e] > probs[best]", "probs[e] >= probs[best]"),
    ("softmax not normalised", "probs[e] /= den;", "probs[e] /= 1.0;"),
    ("router row stride", "dot_bf16(router + (int64_t)e * H, xd, H)", "dot_bf16(router + (int64_t)e, xd, H)"),
    ("silu sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("up uses gate weights", "double u = dot_bf16(wu", "double u = dot_bf16(wg"),
    ("gate without silu", "a[i] = silu(g) * u;", "a[i] = g * u;"),
    ("assignment instead of accumulation", "acc[h] += scale *", "acc[h] = scale *"),
    ("routing weight dropped", "acc[h] += scale * dot_bf16", "acc[h] += dot_bf16"),
    ("shared gate sign", "double gamma = sigmoid(dot_bf16", "double gamma = sigmoid(-dot_bf16"),
    ("shared expert dropped", "        if (J->sg) {", "        if (0) {"),
    ("unstable grouping", "for (int64_t p = 0; p < P; ++p)\n            if (ids[p] == e)",
     "for (int64_t p = P - 1; p >= 0; --p)\n            if (ids[p] == e)"),
    ("offsets not accumulated", "offsets[e + 1] = offsets[e] + counts[e];", "offsets[e + 1] = counts[e];"),
    ("wrong padding sentinel", "(i < c) ? order[offsets[e] + i] : (int32_t)P", "(i < c) ? order[offsets[e] + i] : (int32_t)(P - 1)"),
    ("segments not padded", "int64_t seg = (c + BM - 1) / BM * BM;", "int64_t seg = c;"),
    ("rmsnorm without eps", "double inv = 1.0 / sqrt(ss / H + eps);", "double inv = 1.0 / sqrt(ss / H);"),
    ("rmsnorm sum not averaged", "double inv = 1.0 / sqrt(ss / H + eps);", "double inv = 1.0 / sqrt(ss + eps);"),
    ("gemma weight not offset", "(gemma ? 1.0 + wh : wh)", "(gemma ? wh : wh)"),
    ("residual add dropped", "round_to_bf16(widen_bf16(x[n * H + h]) + widen_bf16(residual[n * H + h]))", "round_to_bf16(widen_bf16(x[n * H + h]))"),
]


def test_unmutated_oracle_passes_every_pin():
    assert pins.failures(oracle.default()) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for '{name}' not unique"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    bad = pins.failures(oracle.Oracle(lib))
    assert bad, f"mutant '{name}' passed every pin"
