"""The oracle's pins catch plausible mistakes: each entry below plants one mistake in a copy of
oracle/rope_causal_oracle.c (a wrong sign, pairing, frequency, mask, head map, scale, log base,
position, stride, decode, or a dropped term of the backward's chain rule), builds it into a
temporary directory, and runs the pin suites against it.  At least one pin must fail for every
mutant; the unmodified oracle passes the same suites in the ordinary test run.

Runs on the CPU only (no GPU, no CUDA path involved).
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_SUITES = ["tests/test_oracle_pins.py", "tests/test_oracle_variant_pins.py",
              "tests/test_oracle_kv_position_pins.py", "tests/test_oracle_bwd_pins.py"]

# name -> list of (original text, planted text); every original must occur exactly once.
MUTANTS = {
    # rotation (half-split form, angles, decode of the inputs)
    "rotation sign of x'[k]": [("y[ia] = a * c - b * s;", "y[ia] = a * c + b * s;")],
    "rotation sign of x'[k+d/2]": [("y[ib] = b * c + a * s;", "y[ib] = b * c - a * s;")],
    "frequency exponent -k/d instead of -2k/d": [("pow(base, -2.0 * (double)k / (double)r)",
                                                  "pow(base, -1.0 * (double)k / (double)r)")],
    "pairs (2k, 2k+1) where (k, k+d/2) is meant": [
        ("int ia = f.interleaved ? 2 * k : k;", "int ia = f.interleaved ? k : 2 * k;"),
        ("int ib = f.interleaved ? 2 * k + 1 : k + half;", "int ib = f.interleaved ? k + half : 2 * k + 1;")],
    "key position off by one": [("double pos = c->kpos ? c->kpos[bj] : (double)j;",
                                 "double pos = c->kpos ? c->kpos[bj] : (double)(j + 1);")],
    "fp16 subnormal scale": [("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);")],
    "bf16 decode shift": [("uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;")],
    # masked softmax attention
    "mask drops the diagonal": [
        ("for (int64_t j = 0; j <= last; ++j) { /* causal", "for (int64_t j = 0; j < last + (last == 0); ++j) { /* causal"),
        ("  for (int64_t j = 0; j <= last; ++j) {\n    score[j] = exp",
         "  for (int64_t j = 0; j < last + (last == 0); ++j) {\n    score[j] = exp"),
        ("  for (int64_t j = 0; j <= last; ++j) {\n    double p = score[j] / denom;",
         "  for (int64_t j = 0; j < last + (last == 0); ++j) {\n    double p = score[j] / denom;")],
    "GQA head map h mod Hkv": [("int hk = h / g; /* GQA", "int hk = h % c->Hkv; /* GQA")],
    "softmax scale missing": [("  double scale = 1.0 / sqrt((double)d);\n  double mx = -INFINITY;\n  for (int64_t j = 0; j <= last; ++j) { /*",
                               "  double scale = 1.0;\n  double mx = -INFINITY;\n  for (int64_t j = 0; j <= last; ++j) { /*")],
    "lse in log2 units": [("= mx + log(denom);", "= mx + log2(denom);")],
    "lse without the max": [("score[j] = exp(score[j] - mx);", "score[j] = exp(score[j]);")],
    "probabilities not normalised": [("double p = score[j] / denom;", "double p = score[j];")],
    # RoPE variants
    "rotary tail not copied": [("for (int e = f.r; e < f.d; ++e) y[e] = x[e];",
                                "for (int e = f.r; e < f.d; ++e) y[e] = 0.0;")],
    "interleaved pair order swapped": [
        ("int ia = f.interleaved ? 2 * k : k;", "int ia = f.interleaved ? 2 * k + 1 : k;"),
        ("int ib = f.interleaved ? 2 * k + 1 : k + half;", "int ib = f.interleaved ? 2 * k : k + half;")],
    "partial rotary pairs (k, k+d/2)": [("int ib = f.interleaved ? 2 * k + 1 : k + half;",
                                         "int ib = f.interleaved ? 2 * k + 1 : k + f.d / 2;")],
    # more keys than queries, explicit positions
    "query i sees keys j <= i with extra keys": [("int64_t last = (int64_t)(c->Nk - c->Nq) + i;",
                                                  "int64_t last = i;")],
    "default query position i": [("c->qpos[(size_t)b * c->Nq + (size_t)i] : (double)last;",
                                  "c->qpos[(size_t)b * c->Nq + (size_t)i] : (double)i;")],
    "dq rotated back at position i": [("c->qpos[(size_t)b * Nq + (size_t)i] : (double)last;",
                                       "c->qpos[(size_t)b * Nq + (size_t)i] : (double)i;")],
    "key positions without the batch stride": [("double pos = c->kpos ? c->kpos[bj] : (double)j;",
                                                "double pos = c->kpos ? c->kpos[j] : (double)j;")],
    "query positions without the batch stride": [("c->qpos[(size_t)b * c->Nq + (size_t)i]", "c->qpos[(size_t)i]")],
    "value rows strided by Nq": [("size_t vbase = (((size_t)b * c->Nk + (size_t)j)",
                                  "size_t vbase = (((size_t)b * c->Nq + (size_t)j)")],
    # backward
    "dS sign": [("double dS = exp(s[j] - mx) / den * (dP[j] - Dsum);",
                 "double dS = exp(s[j] - mx) / den * (Dsum - dP[j]);")],
    "dS without D (key pass)": [("double dS = p * (dP - c->D[st]);", "double dS = p * dP;")],
    "D without P": [("Dsum += exp(s[j] - mx) / den * dP[j];", "Dsum += dP[j];")],
    "dq rotated forward, not back": [("rope_rotate_vec(dqr, out, c->form, -qp, c->theta);",
                                      "rope_rotate_vec(dqr, out, c->form, qp, c->theta);")],
    "dk rotated forward, not back": [("rope_rotate_vec(dkr, c->dk + obase, c->form, -kp, c->theta);",
                                      "rope_rotate_vec(dkr, c->dk + obase, c->form, kp, c->theta);")],
    "dv without P": [("dvj[e] += p * dOi[e];", "dvj[e] += dOi[e];")],
    "dk without the scale": [("dkr[e] += dS * qi[e] * scale;", "dkr[e] += dS * qi[e];")],
    "dq without the scale": [("for (int e = 0; e < d; ++e) dqr[e] += dS * kj[e] * scale;",
                              "for (int e = 0; e < d; ++e) dqr[e] += dS * kj[e];")],
    "key pass skips the diagonal": [("for (int64_t i = first; i < Nq; ++i) {", "for (int64_t i = first + 1; i < Nq; ++i) {")],
    "key pass without the cached queries' offset": [("int64_t first = j - (int64_t)(Nk - Nq);", "int64_t first = j;")],
    "query pass mask without the offset": [("int64_t last = (int64_t)(Nk - Nq) + i;", "int64_t last = i;")],
    "backward query position without the offset": [("(double)(c->pos_off + bn % c->N)", "(double)(bn % c->N)")],
    "key pass sums one head of the group": [("for (int h = hk * g; h < (hk + 1) * g; ++h) {",
                                             "for (int h = hk * g; h < hk * g + 1; ++h) {")],
}


def _mutate(src: str, edits):
    for old, new in edits:
        assert src.count(old) == 1, f"mutation text not found exactly once: {old!r}"
        src = src.replace(old, new)
    return src


def _run_pins(name, edits, tmp):
    with open(oracle.source_path()) as f:
        src = _mutate(f.read(), edits)
    slug = "".join(ch if ch.isalnum() else "_" for ch in name)
    c_path = os.path.join(tmp, f"{slug}.c")
    with open(c_path, "w") as f:
        f.write(src)
    lib = oracle.compile_source(c_path, os.path.join(tmp, f"{slug}.so"))
    env = dict(os.environ, **{oracle.LIB_ENV: lib})
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", *PIN_SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_mutation_text_applies():
    with open(oracle.source_path()) as f:
        src = f.read()
    for name, edits in MUTANTS.items():
        assert _mutate(src, edits) != src, name


def test_each_planted_mistake_fails_a_pin(tmp_path):
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda kv: _run_pins(kv[0], kv[1], str(tmp_path)), MUTANTS.items()))
    survivors = [(name, out) for name, rc, out in results if rc == 0]
    assert not survivors, "planted mistakes that no pin caught: " + "; ".join(n for n, _ in survivors)
    # a failing pin, not a crash of the collection: pytest exits 1 when tests fail
    crashed = [(name, rc, out) for name, rc, out in results if rc not in (1,)]
    assert not crashed, f"mutant runs that did not end in a failing pin: {crashed}"
