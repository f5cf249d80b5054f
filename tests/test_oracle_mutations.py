"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a scratch copy of the oracle's C source (on
the CPU only), rebuilds it, and runs the pin suite against it: the suite has
to fail.  This is the evidence that the pins constrain every step of the
oracle (unpacking, zero point, scale, sign, group and row indexing, operand
order, E2M1 decoding, expert indirection, the symmetric zero point)."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "swap_nibbles": ("(k % 2 == 0) ? (b & 0x0f) : (b >> 4)",
                     "(k % 2 == 0) ? (b >> 4) : (b & 0x0f)"),
    "drop_zero_point": ("float d = q - zf;", "float d = q;"),
    "flip_sign": ("float d = q - zf;", "float d = zf - q;"),
    "drop_scale": ("float w = d * sf;", "float w = d;"),
    "group_index": ("s[n * G + k / g]", "s[n * G + k % G]"),
    "row_index": ("s[n * G + k / g]", "s[k / g]"),
    "e2m1_bias": ("ex - 1)", "ex)"),
    "expert_offset": ("int64_t r = e * N + n;", "int64_t r = n;"),
    "transposed_activation": (
        "acc += (double)w * oracle_bf16_to_f64(X[m * K + k]);",
        "acc += (double)w * oracle_bf16_to_f64(X[m * K + (n % K)]);"),
    "activation_row": ("X[m * K + k]", "X[k]"),
    "symmetric_zero_point": ("z ? (float)oracle_f16_to_f64(z[n * G + k / g]) : 8.0f;\n                float sf",
                             "z ? (float)oracle_f16_to_f64(z[n * G + k / g]) : 7.0f;\n                float sf"),
    "bf16_weight_transposed": ("oracle_bf16_to_f64(W[n * K + k])", "oracle_bf16_to_f64(W[k * N + n])"),
    "moe_gemm_id_index": ("int64_t e = ids[m * topk + j];", "int64_t e = ids[j * M + m];"),
    "moe_gemm_output_row": ("double *y = Y + (m * topk + j) * N;", "double *y = Y + (j * M + m) * N;"),
    "fp4_scale_index": ("s[r * G + k / g]);\n            W[r * K + k] = v * sf;",
                        "s[r * G]);\n            W[r * K + k] = v * sf;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutated_oracle(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(os.path.join(ROOT, "oracle", "w4a16_oracle.c")).read()
    assert before in src, "mutation site missing: " + name
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "*.tmp.*",
                                                  "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copytree(os.path.join(ROOT, "synth"), tmp_path / "synth",
                    ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), tmp_path / "pytest.ini")
    (tmp_path / "oracle" / "w4a16_oracle.c").write_text(src.replace(before, after))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p",
                        "no:cacheprovider", "tests/test_oracle_pins.py"],
                       cwd=tmp_path, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 1, r.stdout[-2000:] + r.stderr[-2000:]
    assert "failed" in r.stdout
