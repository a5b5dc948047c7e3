"""The oracle's pins reject plausible mistakes (CPU only).

Each case copies the oracle's C source, plants one mistake that a careful
restatement of the scheme could still make (a rounding rule, a sign, an
index, a dropped term, a swapped scale), compiles the copy with the
oracle's flags, and runs the CPU pin suites against it: at least one pin
must fail.  An unaltered copy built the same way must pass, so a broken
harness cannot make every mistake look caught."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_e4m3.py", "tests/test_oracle_quant.py", "tests/test_oracle_gemm.py",
        "tests/test_oracle_golden.py", "tests/test_oracle_activation.py"]

# (name, text in the source, replacement)
MUTANTS = [
    ("E4M3 ties away from zero",
     "if (rest > 0x80000u || (rest == 0x80000u && (keep & 1u))) code += 1u;",
     "if (rest >= 0x80000u) code += 1u;"),
    ("E4M3 subnormal ties not to even",
     "if (frac > 0.5f || (frac == 0.5f && (m & 1u))) m += 1u;",
     "if (frac >= 0.5f) m += 1u;"),
    ("E4M3 NaN instead of saturation",
     "if (x >= 448.0f) return (uint8_t)(sign | 0x7e);    /* saturate */",
     "if (x >= 464.0f) return (uint8_t)(sign | 0x7f);"),
    ("E4M3 decode exponent bias off by one",
     "v = ldexp(8.0 + (double)m, e - 7 - 3);",
     "v = ldexp(8.0 + (double)m, e - 8 - 3);"),
    ("BF16 rounding truncates",
     "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;",
     "/* truncated */"),
    ("scale is 448/amax",
     "*s = va / 448.0f;",
     "*s = 448.0f / va;"),
    ("all-zero tile scale 0",
     "*s = 1.0f;\n        *inv = 1.0f;",
     "*s = 0.0f;\n        *inv = 1.0f;"),
    ("row-wise payload divided by the multiplier",
     "q[r * cols + b * 128 + i] = orc_e4m3_encode(orc_bf16_to_f32(t[i]) * inv);",
     "q[r * cols + b * 128 + i] = orc_e4m3_encode(orc_bf16_to_f32(t[i]) * sc);"),
    ("128x1 amax along the row",
     "float a = fabsf(orc_bf16_to_f32(x[(b * 128 + i) * cols + c]));",
     "float a = fabsf(orc_bf16_to_f32(x[(b * 128) * cols + (c + i) % cols]));"),
    ("token-tail padding payload not zero",
     "i < n ? orc_e4m3_encode(orc_bf16_to_f32(x[(b * 128 + i) * cols + c]) * inv) : 0x00;",
     "i < n ? orc_e4m3_encode(orc_bf16_to_f32(x[(b * 128 + i) * cols + c]) * inv) : 0x38;"),
    ("W^T written in W's layout",
     "if (qT) qT[c * n + r] = code;",
     "if (qT) qT[r * k + c] = code;"),
    ("promotion ignores the B scale",
     "float scale = sa[j * sa_stride] * sb[j * sb_stride];",
     "float scale = sa[j * sa_stride];"),
    ("promotion as multiply then add",
     "acc = fmaf((float)p, scale, acc);",
     "acc = (float)p * scale + acc;"),
    ("promotion over blocks in reverse order",
     "for (int64_t j = 0; j < kc / 128; j++) {\n        double p = 0.0, pabs = 0.0;",
     "for (int64_t j = kc / 128 - 1; j >= 0; j--) {\n        double p = 0.0, pabs = 0.0;"),
    ("dgrad reads W transposed",
     "for (int64_t n = 0; n < N; n++) col[n] = wq[n * K + k]; /* column k of W */",
     "for (int64_t n = 0; n < N; n++) col[n] = wq[k * N + n]; /* column k of W */"),
    ("SiLU with e^+g",
     "float t = orc_exp_cw(-g);",
     "float t = orc_exp_cw(g);"),
    ("e^x polynomial without its r^2/2 term",
     "p = fmaf(p, r, 0.5f);",
     "p = fmaf(p, r, 0.0f);"),
    ("row-wise amax of signed values",
     "float a = fabsf(orc_bf16_to_f32(t[i]));",
     "float a = orc_bf16_to_f32(t[i]);"),
    ("weight amax over the block's first column only",
     "float a = fabsf(orc_bf16_to_f32(w[(bn * 128 + i) * k + bk * 128 + j]));",
     "float a = fabsf(orc_bf16_to_f32(w[(bn * 128 + i) * k + bk * 128]));"),
    ("row-wise scales stored row-major",
     "            s[b * mp + r] = sc;",
     "            s[r * nb + b] = sc;"),
    ("128x1 scales stored column-major",
     "sT[b * cols + c] = sc;",
     "sT[c * nb + b] = sc;"),
    ("weight scales stored transposed",
     "s[bn * nbk + bk] = sc;",
     "s[bk * nbn + bn] = sc;"),
    ("E4M3 drops the sign of a value that rounds to zero",
     "        return (uint8_t)(sign | m);",
     "        return (uint8_t)(m ? (sign | m) : 0u);"),
    ("wgrad applies the row scale twice",
     "sdyt + n, N,\n                                  sxt + k, K, &sabs);",
     "sdyt + n, N,\n                                  sdyt + n, N, &sabs);"),
    ("dgrad weight scale of the transposed block",
     "sw + k / 128, kb, &sabs);",
     "sw + (k / 128) * kb, 1, &sabs);"),
    ("e^x without the low part of ln 2",
     "    r = fmaf(-n, LN2_LO_F, r);\n",
     ""),
    ("SiLU rounds g / (1 + e^-g) to BF16 before the product",
     "    float sg = g / d;\n",
     "    float sg = orc_bf16_to_f32(orc_f32_to_bf16(g / d));\n"),
]


def build_copy(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(src), "-o", str(lib), "-lm"])
    return str(lib)


def run_pins(lib):
    env = dict(os.environ, FP8BS_ORACLE_LIB=lib)
    return subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unaltered_copy_passes(tmp_path):
    lib = build_copy(tmp_path, "unaltered", open(oracle.SOURCE).read())
    r = run_pins(lib)
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, find, repl):
    text = open(oracle.SOURCE).read()
    assert text.count(find) == 1, f"the source no longer holds the line this case alters: {find!r}"
    lib = build_copy(tmp_path, "mutant", text.replace(find, repl))
    r = run_pins(lib)
    assert r.returncode != 0, f"no pin failed with the mistake '{name}' planted"
