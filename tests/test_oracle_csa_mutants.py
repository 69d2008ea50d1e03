"""Mutation check of the attention consumer oracle's pins: each mutant plants
one plausible mistake in a copy of oracle/csa.py (in a temporary directory);
the pin suite must fail on every one of them."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "csa.py")

MUTANTS = {
    "scale-dropped": ("s = scale * (kv @ q.T)", "s = kv @ q.T"),
    "softmax-over-heads": ("m = s.max(axis=0)                      # [H]\n    p = np.exp(s - m)",
                           "m = s.max(axis=1, keepdims=True)\n    p = np.exp(s - m)"),
    "max-not-subtracted": ("p = np.exp(s - m)                      # [n, H]", "p = np.exp(s)"),
    "not-normalised": ("o = (p.T @ kv) / l[:, None]", "o = p.T @ kv"),
    "lse-log2": ("return o, m + np.log(l)", "return o, m + np.log2(l)"),
    "lse-without-max": ("return o, m + np.log(l)", "return o, np.log(l)"),
    "holes-kept": ("js = js[js >= 0]\n        o, lse", "o, lse"),
    "bf16-low-half": ("<< 16).view(np.float32)", "<< 15).view(np.float32)"),
    "row-stride-512": ("at = kv_offset + (int(j) % R) * 1024", "at = kv_offset + (int(j) % R) * 512"),
    "page-of-request-0": ("page = int(block_table[b, int(j) // R])",
                          "page = int(block_table[0, int(j) // R])"),
    "values-are-queries": ("o = (p.T @ kv) / l[:, None]", "o = (p.T @ (kv * 0 + q.mean(0))) / l[:, None]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_kill_mutant(name, tmp_path):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation anchor not found: %s" % name
    mut = tmp_path / "csa_mut.py"
    mut.write_text(src.replace(old, new))
    env = dict(os.environ, CSA_ORACLE_PATH=str(mut))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-W", "ignore", os.path.join(ROOT, "tests", "test_oracle_csa_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])


def test_control_copy_passes(tmp_path):
    mut = tmp_path / "csa_copy.py"
    mut.write_text(open(SRC).read())
    env = dict(os.environ, CSA_ORACLE_PATH=str(mut))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-W", "ignore", os.path.join(ROOT, "tests", "test_oracle_csa_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
