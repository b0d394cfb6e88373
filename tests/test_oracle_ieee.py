"""Pins of the oracle's IEEE arithmetic (conversions and the per-hop add).

The oracle rounds binary32 to binary16 / bfloat16 with its own bit-level code.
These tests compare it with arithmetic the oracle does not contain, over whole
input spaces (every binary32 encoding, every pair of 16-bit encodings, on all
host cores): the C compiler's ``_Float16`` / ``__bf16`` casts and an exact
binary64 sum rounded once; plus numpy's float16 conversion and torch's
bfloat16 conversion on samples.  tests/test_ieee_gpu.py pins the same
conversions and hops against the GPU's.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def pin_exe(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("pin") / "pin_ieee")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp",
                    "-I", os.path.join(ROOT, "oracle"), os.path.join(HERE, "csrc", "pin_ieee.c"),
                    os.path.join(ROOT, "oracle", "ring_oracle.c"), "-lm", "-o", exe], check=True)
    return exe


def run_pin(exe, test, lo=0, hi=0):
    out = subprocess.run([exe, test, str(lo), str(hi), "1"], check=True,
                         capture_output=True, text=True).stdout.split()
    assert out[0] == test
    checked, bad, first = int(out[1]), int(out[2]), int(out[3])
    assert checked > 0
    assert bad == 0, f"{test}: {bad} mismatches of {checked}, first at input {first:#x}"
    return checked


FULL = 1 << 32  # every binary32 encoding; every pair of 16-bit encodings


def test_widening_exhaustive(pin_exe):
    assert run_pin(pin_exe, "f16_to_f32") == 65536
    assert run_pin(pin_exe, "bf16_to_f32") == 65536


def test_f32_to_f16_rounding_exhaustive(pin_exe):
    # all 2^32 binary32 encodings against the compiler's (_Float16) cast
    assert run_pin(pin_exe, "f32_to_f16", 0, FULL) == FULL


def test_f32_to_bf16_rounding_exhaustive(pin_exe):
    assert run_pin(pin_exe, "f32_to_bf16", 0, FULL) == FULL


def test_hop_add_f16_exhaustive(pin_exe):
    # one hop = binary32 sum rounded once to binary16; every one of the 2^32
    # pairs against the exact (binary64) sum rounded once by the compiler
    assert run_pin(pin_exe, "add_f16", 0, FULL) == FULL


def test_hop_add_bf16_exhaustive(pin_exe):
    assert run_pin(pin_exe, "add_bf16", 0, FULL) == FULL


def test_hop_add_f32(pin_exe):
    # binary32 pairs number 2^64, beyond any exhaustive run: 2^24 pairs drawn
    # by a fixed mixing function cover every exponent and sign combination
    run_pin(pin_exe, "add_f32", 0, 1 << 24)


def test_f16_against_numpy(orc):
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(1 << 18).astype(np.float32) * 1e-3,
                        rng.standard_normal(1 << 18).astype(np.float32) * 3e4,
                        np.array([0.0, -0.0, np.inf, -np.inf, 65504.0, 65520.0, 65519.996,
                                  2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26],
                                 dtype=np.float32)])
    mine = orc.f32_to_wire(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(mine, ref)


def test_bf16_against_torch(orc):
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.standard_normal(1 << 18).astype(np.float32),
                        (rng.standard_normal(1 << 16) * 1e-39).astype(np.float32),
                        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4028235e38],
                                 dtype=np.float32)])
    mine = orc.f32_to_wire(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, ref)


def test_f16_hop_against_numpy_add(orc):
    # numpy's float16 addition is correctly rounded: it must equal one oracle hop
    rng = np.random.default_rng(13)
    a = (rng.standard_normal(1 << 18) * 1e-3).astype(np.float16)
    b = (rng.standard_normal(1 << 18) * 1e-3).astype(np.float16)
    mine = orc.wire_add(a.view(np.uint16), b.view(np.uint16), "f16")
    np.testing.assert_array_equal(mine, (a + b).view(np.uint16))
