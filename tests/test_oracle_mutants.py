"""Each plausible mistake planted in the oracle's C source must fail a pin.

The mutant is compiled on the CPU into a temporary library and the pin suite
(test_oracle_pins.py) runs against it in a child process; the child must
report a failure.  This shows the pins constrain every step of the oracle:
window choice, record layout, planes, decode, the 8-bit view, the fp64 GEMM
and its bound, argmax ties, tree acceptance, the two-level-verification splice, the
node budget, the INT8 head's quantizer, bound and certified argmax, and the gated
delta rule's path verify, commit and three-piece split.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "w12_oracle.c")

MUTANTS = {
    "window ties go high": ("if (count > best_count) {", "if (count >= best_count) {"),
    "window range short": ("for (int b = 1; b <= 239; ++b) {", "for (int b = 1; b <= 238; ++b) {"),
    "window 15 binades": ("for (int E = b; E <= b + 15; ++E) count += hist[E];",
                          "for (int E = b; E <= b + 14; ++E) count += hist[E];"),
    "record drops sign": ("r = (s << 11) | (eo << 7) | m;", "r = (eo << 7) | m;"),
    "record sign misplaced": ("r = (s << 11) | (eo << 7) | m;", "r = (s << 10) | (eo << 7) | m;"),
    "lo nibble order swapped": ("lo[n * lo_row + k / 2] |= (uint8_t)((r & 0xFu) << ((k & 1) ? 4 : 0));",
                                "lo[n * lo_row + k / 2] |= (uint8_t)((r & 0xFu) << ((k & 1) ? 0 : 4));"),
    "decode exponent off by one": ("((base[n] + eo) << 7)", "((base[n] + eo + 1) << 7)"),
    "q8 rounds up": ("uint32_t r = q8 ? ((uint32_t)hi[n * K + k] << 4)", "uint32_t r = q8 ? (((uint32_t)hi[n * K + k] << 4) | 8u)"),
    "escape drops sign": ("esc[n_esc] = ((uint32_t)k << 16) | w;", "esc[n_esc] = ((uint32_t)k << 16) | (w & 0x7FFFu);"),
    "gemm reversed k": ("double p = bf16_value(x[m * K + k]) * bf16_value(W[n * K + k]);",
                        "double p = bf16_value(x[m * K + (K - 1 - k)]) * bf16_value(W[n * K + k]);"),
    "gemm sign flip": ("acc += p;", "acc -= p;"),
    "gemm bound signed": ("mag += p < 0 ? -p : p;", "mag += p;"),
    "argmax ties go high": ("  return a > b;\n}", "  return a >= b;\n}"),
    "accept compares own token": ("acc[i] = acc[p] && draft[i] == tok[p];", "acc[i] = acc[p] && draft[i] == tok[i];"),
    "accept ignores parent": ("acc[i] = acc[p] && draft[i] == tok[p];", "acc[i] = draft[i] == tok[p];"),
    "accept depth ties go high": ("if (acc[i] && depth[i] > depth[best]) best = i;",
                                  "if (acc[i] && depth[i] >= depth[best]) best = i;"),
    "bonus from parent": ("*bonus = tok[best];", "*bonus = tok[parent[best] < 0 ? 0 : parent[best]];"),
    "splice bonus under the wrong node": ("  parent[L + 1] = L;", "  parent[L + 1] = L > 0 ? L - 1 : L;"),
    "splice path drafts by position": ("    draft[i] = draft_q[path[i]];", "    draft[i] = draft_q[i];"),
    "splice subtree parents not shifted": ("parent[i] = sub_parent[j] < 0 ? L + 1 : L + 2 + sub_parent[j];",
                                           "parent[i] = sub_parent[j] < 0 ? L + 1 : L + 1 + sub_parent[j];"),
    "splice new rows off by one": ("    src[i] = -1 - (j + 1);", "    src[i] = -1 - j;"),
    "splice drops the bonus token": ("  draft[L + 1] = bonus;", "  draft[L + 1] = draft_q[path[L]];"),
    "budget scores add": ("score[i] = score[off[r] + p] * conf[i];", "score[i] = score[off[r] + p] + conf[i];"),
    "budget deeper first on ties": ("(depth[j] < depth[i] || (depth[j] == depth[i] && j < i))",
                                    "(depth[j] > depth[i] || (depth[j] == depth[i] && j < i))"),
    "budget per request ignored": ("if (j == i || (per_request && req[j] != req[i])) continue;",
                                   "if (j == i) continue;"),
    "budget parents not renumbered": ("parent_out[kept + n] = i == off[r] ? -1 : newidx[off[r] + parent[i]];",
                                      "parent_out[kept + n] = i == off[r] ? -1 : parent[i];"),
    "budget keeps one too many": ("      keep[i] = rank < budget;", "      keep[i] = rank <= budget;"),
    "i8 scale off 128": ("const float s = amax / 127.0f;", "const float s = amax / 128.0f;"),
    "i8 codes truncate": ("q = rint(w / (double)s);", "q = trunc(w / (double)s);"),
    "i8 codes round half up": ("q = rint(w / (double)s);", "q = floor(w / (double)s + 0.5);"),
    "i8 sign bit dropped": ("code[n * K + k] = (uint8_t)((iq < 0 ? 0x80 : 0x00) | (iq < 0 ? -iq : iq));",
                            "code[n * K + k] = (uint8_t)(iq < 0 ? -iq : iq);"),
    "i8 bound drops the quantization error": ("cbound[n] = round_up_float(sqrt(e2) + gamma * (double)s * sqrt(q2));",
                                              "cbound[n] = round_up_float(gamma * (double)s * sqrt(q2));"),
    "i8 bound halves the quantization error": ("cbound[n] = round_up_float(sqrt(e2) + gamma * (double)s * sqrt(q2));",
                                               "cbound[n] = round_up_float(0.5 * sqrt(e2) + gamma * (double)s * sqrt(q2));"),
    "cert threshold uses the upper end": ("      if (lo[v] > thr) thr = lo[v];", "      if (hi[v] > thr) thr = hi[v];"),
    "cert keeps only the approximate argmax": ("      if (hi[v] < thr) continue;", "      if (hi[v] < thr || lo[v] < thr) continue;"),
    "cert ties go high": ("      if (best < 0 || better(L, best_val)) {", "      if (best < 0 || !better(best_val, L)) {"),
    "split truncates": ("  u += 0x7FFFu + ((u >> 16) & 1u);\n  return (uint16_t)(u >> 16);\n}\n\nstatic float bf16_float",
                        "  return (uint16_t)(u >> 16);\n}\n\nstatic float bf16_float"),
    "split drops the third piece": ("    s3[i] = bf16_rne_bits(r2);", "    s3[i] = 0;"),
    "gdn gate dropped": ("S[r * dk + c] = alpha * S[r * dk + c] + coef * bf16_value(k[c]);",
                         "S[r * dk + c] = S[r * dk + c] + coef * bf16_value(k[c]);"),
    "gdn erase not gated": ("const double coef = beta * bf16_value(v[r]) - alpha * beta * u;",
                            "const double coef = beta * bf16_value(v[r]) - beta * u;"),
    "gdn write sign flipped": ("const double coef = beta * bf16_value(v[r]) - alpha * beta * u;",
                               "const double coef = -beta * bf16_value(v[r]) - alpha * beta * u;"),
    "gdn path includes the root": ("for (int64_t j = i; j > 0; j = parent[j]) path[L++] = j;",
                                   "for (int64_t j = i; j >= 0; j = parent[j]) path[L++] = j;"),
    "gdn path applied backwards": ("      for (int64_t t = L - 1; t >= 0; --t) {\n        const int64_t j = path[t];",
                                   "      for (int64_t t = 0; t < L; ++t) {\n        const int64_t j = path[t];"),
    "gdn output reads the key": ("o += S[r * dk + c] * bf16_value(q[(i * H + h) * dk + c]);",
                                 "o += S[r * dk + c] * bf16_value(k[(i * H + h) * dk + c]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {name}"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", str(so), str(mut)])
    env = dict(os.environ, W12_ORACLE_SO=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant '{name}' survived the pins:\n{r.stdout[-2000:]}"
