"""The oracle's pins catch plausible mistakes: each case plants one mistake in a copy of
the oracle's C source (a dropped term, a wrong sign, index or bit position, swapped or
transposed operands), rebuilds the copy and runs the pins of test_oracle.py against it;
at least one pin must fail. Nothing here touches the real oracle or the CUDA path."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, statement in oracle.c, the same statement with the mistake planted)
MUTANTS = [
    ("q4_k min term dropped",
     "w[b * 256 + e] = a * (float)q - c;\n                }\n            }\n        } else if (fmt == OR_Q5_K)",
     "w[b * 256 + e] = a * (float)q;\n                }\n            }\n        } else if (fmt == OR_Q5_K)"),
    ("q4_k scale and min fields swapped",
     "int sc = q4k_field(blk + 4, j), m = q4k_field(blk + 4, 8 + j);\n                    int q = (blk[16",
     "int sc = q4k_field(blk + 4, 8 + j), m = q4k_field(blk + 4, j);\n                    int q = (blk[16"),
    ("q4_k nibble order",
     "int q = (blk[16 + e / 2] >> (4 * (e & 1))) & 15;",
     "int q = (blk[16 + e / 2] >> (4 * (1 - (e & 1)))) & 15;"),
    ("q4_k sub-blocks of 16",
     "                    int j = e / 32;\n                    int sc = q4k_field(blk + 4, j), m = q4k_field(blk + 4, 8 + j);\n"
     "                    int q = (blk[16",
     "                    int j = (e / 16) & 7;\n                    int sc = q4k_field(blk + 4, j), m = q4k_field(blk + 4, 8 + j);\n"
     "                    int q = (blk[16"),
    ("q5_k fifth bit taken column-wise",
     "int hi = (blk[16 + e / 8] >> (e & 7)) & 1;",
     "int hi = (blk[16 + (e & 31)] >> (e / 32)) & 1;"),
    ("q5_k fifth bit weighted 8",
     "int q = lo | (hi << 4);\n                    float a = d * (float)sc;\n                    float c",
     "int q = lo | (hi << 3);\n                    float a = d * (float)sc;\n                    float c"),
    ("q6_k offset sign", "w[b * 256 + e] = a * (float)(q - 32);", "w[b * 256 + e] = a * (float)(q + 32);"),
    ("q6_k scales unsigned", "int sc = (int8_t)blk[192 + e / 16];", "int sc = (uint8_t)blk[192 + e / 16];"),
    ("q6_k one scale per 32", "int sc = (int8_t)blk[192 + e / 16];", "int sc = (int8_t)blk[192 + e / 32];"),
    ("q8_0 quants unsigned", "w[b * 32 + i] = d * (float)(int8_t)blk[2 + i];", "w[b * 32 + i] = d * (float)blk[2 + i];"),
    ("nvfp4 tensor scale dropped", "W[r * K + k] = p * sT;", "W[r * K + k] = p;"),
    ("nvfp4 one block scale per 32", "float sb = or_e4m3_to_f32(scales[r * (K / 16) + k / 16]);",
     "float sb = or_e4m3_to_f32(scales[r * (K / 16) + k / 32]);"),
    ("fp8 row scale indexed by column", "W[r * K + k] = or_e4m3_to_f32(canon[r * K + k]) * s;",
     "W[r * K + k] = or_e4m3_to_f32(canon[r * K + k]) * rdf32(canon + rows * K + 4 * (k % rows));"),
    ("gemv with W transposed",
     "double p = (double)W[n * K + k] * (double)or_bf16_to_f32(x_bf16[m * K + k]);",
     "double p = (double)W[k * N % (N * K) + n] * (double)or_bf16_to_f32(x_bf16[m * K + k]);"),
    ("gemv drops the last k", "for (int64_t k = 0; k < K; k++) {\n                double p",
     "for (int64_t k = 0; k < K - 1; k++) {\n                double p"),
    ("error scale signed", "ab += fabs(p);", "ab += p;"),
    ("silu sign", "h[i] = (g[i] / (1.0 + exp(-g[i]))) * u[i];", "h[i] = (g[i] / (1.0 + exp(g[i]))) * u[i];"),
    ("gate and up swapped", "h[i] = (g[i] / (1.0 + exp(-g[i]))) * u[i];", "h[i] = (u[i] / (1.0 + exp(-u[i]))) * g[i];"),
    ("activation block scale 1.5x too small", "or_f32_to_e4m3(amax / t) : 0;\n            scales[m",
     "or_f32_to_e4m3(amax / (t / 1.5f)) : 0;\n            scales[m"),
    ("activation nibble order", "codes[m * (K / 2) + e / 2] |= (uint8_t)(c << (4 * (e & 1)));",
     "codes[m * (K / 2) + e / 2] |= (uint8_t)(c << (4 * (1 - (e & 1))));"),
    ("distinct experts sorted descending", "while (j >= 0 && out[j] > v)", "while (j >= 0 && out[j] < v)"),
    ("w4a4 takes the raw activations",
     "a[k] = (double)or_e2m1_to_f32(c) * (double)or_e4m3_to_f32(scales[m * (K / 16) + k / 16]) *\n"
     "                   (double)x_scale;",
     "a[k] = (double)or_bf16_to_f32(x_bf16[m * K + k]) + 0.0 * (double)c * (double)scales[0] *\n"
     "                   (double)x_scale;"),
    ("w4a4 static scale dropped",
     "a[k] = (double)or_e2m1_to_f32(c) * (double)or_e4m3_to_f32(scales[m * (K / 16) + k / 16]) *\n"
     "                   (double)x_scale;",
     "a[k] = (double)or_e2m1_to_f32(c) * (double)or_e4m3_to_f32(scales[m * (K / 16) + k / 16]) *\n"
     "                   1.0;"),
    ("w4a4 error scale signed", "                ab += fabs(t);", "                ab += t;"),
    ("iq4_xs scale offset sign", "float a = d * (float)(ls - 32);\n                W[r * K + b * 256 + e]",
     "float a = d * (float)(32 - ls);\n                W[r * K + b * 256 + e]"),
    ("iq4_xs scale nibble order", "int ls = ((blk[4 + j / 2] >> (4 * (j & 1))) & 15)",
     "int ls = ((blk[4 + j / 2] >> (4 * (1 - (j & 1)))) & 15)"),
    ("iq4_xs scale high bits one per bit", "(((sh >> (2 * j)) & 3) << 4);\n                int q",
     "(((sh >> j) & 3) << 4);\n                int q"),
    ("iq4_xs index nibble order", "int q = (blk[8 + e / 2] >> (4 * (e & 1))) & 15;\n                float a = d * (float)(ls",
     "int q = (blk[8 + e / 2] >> (4 * (1 - (e & 1)))) & 15;\n                float a = d * (float)(ls"),
    ("iq4_xs sub-blocks of 16", "                int j = e / 32;\n                int ls = ((blk[4",
     "                int j = (e / 16) & 7;\n                int ls = ((blk[4"),
    ("int8-dot scale over 128", "float d = amax / 127.0f;\n            scales[m * (K / 32) + b] = d;",
     "float d = amax / 128.0f;\n            scales[m * (K / 32) + b] = d;"),
    ("int8-dot codes truncated", "(int)clampf(rintf(xv[i] / d), -127.0f, 127.0f)",
     "(int)clampf(xv[i] / d, -127.0f, 127.0f)"),
    ("int8-dot raw activations", "for (int64_t k = 0; k < K; k++) a[k] = (double)scales[m * (K / 32) + k / 32] * (double)codes[m * K + k];",
     "for (int64_t k = 0; k < K; k++) a[k] = (double)or_bf16_to_f32(x_bf16[m * K + k]) + 0.0 * codes[0];"),
    ("iq3_s index bit 8 from the next group",
     "idx = blk[2 + g] | (((blk[66 + g / 8] >> (g & 7)) & 1) << 8);",
     "idx = blk[2 + g] | (((blk[66 + (g + 1) % 64 / 8] >> ((g + 1) & 7)) & 1) << 8);"),
    ("iq3_s sign bits per group", "sg = (blk[74 + e / 8] >> (e & 7)) & 1;", "sg = (blk[74 + g / 8] >> (g & 7)) & 1;"),
    ("iq3_s even scales", "float a = d * (float)(2 * sc + 1);\n                float m",
     "float a = d * (float)(2 * sc);\n                float m"),
    ("iq2_s index bits 8..9 one bit apart", "idx = blk[2 + g] | (((blk[66 + g / 4] >> (2 * (g & 3))) & 3) << 8);",
     "idx = blk[2 + g] | (((blk[66 + g / 8] >> (g & 7)) & 3) << 8);"),
    ("iq2_s sign bit order", "sg = (blk[34 + g] >> i) & 1;", "sg = (blk[34 + g] >> (7 - i)) & 1;"),
    ("iq2_s scales per 32 values", "int g = e / gw, i = e % gw, k = e / sbs;",
     "int g = e / gw, i = e % gw, k = e / (2 * sbs);"),
    ("grid entries read column-wise", "float m = (float)G[idx * gw + i];", "float m = (float)G[i * 512 + idx % 512];"),
    ("iq4_xs codebook read before the blocks", "const int8_t* cb = (const int8_t*)(canon + rows * (K / 256) * 136);",
     "const int8_t* cb = (const int8_t*)(canon);"),
]


def _copy(dst):
    os.makedirs(dst / "tests")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), dst / "tests" / "golden")
    for f in ("tests/test_oracle.py", "tests/conftest.py", "synth.py"):
        shutil.copy(os.path.join(ROOT, f), dst / f)


@pytest.mark.parametrize("name,good,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, good, bad, tmp_path):
    _copy(tmp_path)
    src = tmp_path / "oracle" / "oracle.c"
    text = src.read_text()
    assert text.count(good) == 1, f"the statement for '{name}' is no longer in oracle.c"
    src.write_text(text.replace(good, bad))
    r = subprocess.run([sys.executable, "-c", "import oracle; oracle.build()"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle.py"], cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode == 1, f"no pin caught '{name}':\n{r.stdout[-2000:]}"


def test_unmodified_copy_passes(tmp_path):
    # the control: the copied pins pass on the copied oracle as it stands, so a failure
    # above is the planted mistake's doing and not the copy's
    _copy(tmp_path)
    r = subprocess.run([sys.executable, "-c", "import oracle; oracle.build()"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "tests/test_oracle.py"],
                       cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-2000:]
