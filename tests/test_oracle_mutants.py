"""Mutation check of the oracle's pins: each mutant plants one plausible
mistake in a copy of oracle/qli_oracle.c (or oracle/qli_quant_oracle.c) (built on the CPU into a temporary
directory, never touching the real oracle); the pin suite must fail on every
one of them. This shows the pins constrain each step of the definition."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qli_oracle.c")

MUTANTS = {
    "relu-dropped": ("float r = x > 0.0f ? x : 0.0f;", "float r = x;"),
    "divisor-1000": ("(float)s / 1024.0f", "(float)s / 1000.0f"),
    "x-not-rounded": ("float x = oracle_f16_to_f32(oracle_f32_to_f16((float)s / 1024.0f));",
                      "float x = (float)s / 1024.0f;"),
    "product-not-rounded": ("return f16_mul(r, wq);", "return r * wq;"),
    "wq-not-rounded": ("float wq = f16_mul(oracle_f16_to_f32(w_bits), oracle_f16_to_f32(qs_bits));",
                       "float wq = oracle_f16_to_f32(w_bits) * oracle_f16_to_f32(qs_bits);"),
    "k-scale-dropped": ("return acc * oracle_f16_to_f32(k_scale(in, b, j));", "return acc;"),
    "acc-in-fp16": ("acc = acc + oracle_head_term(",
                    "acc = oracle_f16_to_f32(oracle_f32_to_f16(acc)) + oracle_head_term("),
    "visible-off-by-one": ("int64_t seen = pos + 1;", "int64_t seen = pos;"),
    "residual-ignored": ("int64_t S = k_len * ratio + res;", "int64_t S = k_len * ratio;"),
    "dot-index-shift": ("s += (int32_t)qh[d] * (int32_t)k[d];",
                        "s += (int32_t)qh[d] * (int32_t)k[(d + 1) % D];"),
    "weight-head-0": ("in->head_weights[(int64_t)t * in->N + h]",
                      "in->head_weights[(int64_t)t * in->N]"),
    "tie-break-reversed": ("return (a->id > b->id) - (a->id < b->id);",
                           "return (a->id < b->id) - (a->id > b->id);"),
    "last-block-not-pinned": ("bl[C - 1].id = nb - 1;      /* the pinned last visible block */",
                              ";"),
    "block-max-is-min": ("if (sc[j] > m) m = sc[j];", "if (sc[j] < m) m = sc[j];"),
    "consumer-block-16": ("if (in_set && !in_set[j / 8]) continue;",
                          "if (in_set && !in_set[j / 16]) continue;"),
    "output-not-sorted": ("qsort(ids, (size_t)take, sizeof(int64_t), ascending_i64);", ";"),
    "scale-row-wrong": ("memcpy(&bits, in->cache + page * in->page_stride + in->scale_offset + row * 2, 2);",
                        "memcpy(&bits, in->cache + page * in->page_stride + in->scale_offset, 2);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_kill_mutant(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation anchor not found: %s" % name
    mut = tmp_path / "qli_oracle_mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", str(mut), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])


# ---- the query quantiser and index-K writer (qli_quant_oracle.c) -----------

QSRC = os.path.join(ROOT, "oracle", "qli_quant_oracle.c")

QUANT_MUTANTS = {
    "divisor-128": ("row_scale(x, D, 127.0f, &s)", "row_scale(x, D, 128.0f, &s)"),
    "scale-not-fp16": ("const float sf = (float)s;", "const float sf = (float)s * 1.0001f;"),
    "floor-not-round": ("float r = rintf(oracle_bf16_to_f32(x[d]) / sf);",
                        "float r = floorf(oracle_bf16_to_f32(x[d]) / sf);"),
    "clamp-at-128": ("if (r < -127.0f) r = -127.0f;", "if (r < -128.0f) r = -128.0f;"),
    "no-saturation": ("if (isinf((float)s)) s = (_Float16)65504.0f;", ";"),
    "amax-signed": ("const float a = fabsf(v);", "const float a = v;"),
    "row-from-slot-div": ("const int64_t page = m / R, row = m % R;",
                          "const int64_t page = m % R, row = m / R;"),
    "scale-stride-1": ("memcpy(p + scale_offset + row * 2, &s, 2);",
                       "memcpy(p + scale_offset + row, &s, 2);"),
    "padding-written": ("const int64_t m = slot[i];", "const int64_t m = slot[i] < 0 ? 0 : slot[i];"),
}


@pytest.mark.parametrize("name", sorted(QUANT_MUTANTS))
def test_quant_pins_kill_mutant(name, tmp_path):
    src = open(QSRC).read()
    old, new = QUANT_MUTANTS[name]
    assert src.count(old) == 1, "mutation anchor not found: %s" % name
    mut = tmp_path / "qli_quant_oracle_mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libqmut.so"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", SRC, str(mut), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_quant_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])


# ---- the FP8 variant (quant mode 1), both sources --------------------------

FP8_MUTANTS = {
    # (file, anchor, replacement)
    "e4m3-bias-8": (SRC, "else v = ldexp(8.0 + m, e - 10);", "else v = ldexp(8.0 + m, e - 11);"),
    "e4m3-subnormal-as-zero": (SRC, "if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = 0.0;"),
    "fp8-dot-in-float": (SRC, "    double s = 0.0;\n    for (int32_t d = 0; d < D; ++d) s += oracle_e4m3_to_f64",
                         "    float s = 0.0f;\n    for (int32_t d = 0; d < D; ++d) s += oracle_e4m3_to_f64"),
    "fp8-divisor-1000": (SRC, "oracle_f32_to_f16(s / 1024.0f));", "oracle_f32_to_f16(s / 1000.0f));"),
    "fp8-reads-int8": (SRC, "if (in->quant_mode == 1)\n", "if (in->quant_mode == 3)\n"),
    "e4m3-ties-away": (QSRC, "double n = nearbyint(a / quantum);", "double n = round(a / quantum);"),
    "e4m3-saturates-to-nan": (QSRC, "if (a >= 448.0) return sign | 0x7E;",
                              "if (a >= 448.0) return sign | 0x7F;"),
    "fp8-scale-127": (QSRC, "row_scale(x, D, 448.0f, &s)", "row_scale(x, D, 127.0f, &s)"),
    "fp8-divides-by-another-scale": (QSRC, "const float s8 = (float)s;",
                                     "const float s8 = (float)s * 1.0001f;"),
}


def _fp8_pins(tmp_path, main_src, quant_src):
    lib = tmp_path / "libfp8.so"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", str(main_src), str(quant_src), "-o", str(lib), "-lm"],
                   check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_fp8_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unmutated_builds_pass_their_pins(tmp_path):
    # the harness itself: the sources built the way the mutants are built
    # load and pass, so a killed mutant is killed by a pin
    r = _fp8_pins(tmp_path, SRC, QSRC)
    assert r.returncode == 0, r.stdout[-2000:]
    lib = tmp_path / "libplain.so"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", SRC, "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(FP8_MUTANTS))
def test_fp8_pins_kill_mutant(name, tmp_path):
    path, old, new = FP8_MUTANTS[name]
    src = open(path).read()
    assert src.count(old) == 1, "mutation anchor not found: %s" % name
    mut = tmp_path / os.path.basename(path)
    mut.write_text(src.replace(old, new))
    main_src, quant_src = (mut, QSRC) if path == SRC else (SRC, mut)
    r = _fp8_pins(tmp_path, main_src, quant_src)
    assert r.returncode != 0, "mutant %s survived the FP8 pins:\n%s" % (name, r.stdout[-2000:])
