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
                    "-ffp-contract=off", str(mut), "-o", str(lib)], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])


# ---- the query quantiser and index-K writer (qli_quant_oracle.c) -----------

QSRC = os.path.join(ROOT, "oracle", "qli_quant_oracle.c")

QUANT_MUTANTS = {
    "divisor-128": ("const float quotient = amax / 127.0f;", "const float quotient = amax / 128.0f;"),
    "scale-not-fp16": ("const float sf = (float)s;", "const float sf = quotient;"),
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
