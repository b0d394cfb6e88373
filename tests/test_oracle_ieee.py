"""Pins of the oracle's IEEE arithmetic (conversions and the per-hop add).

The oracle rounds binary32 to binary16 / bfloat16 with its own bit-level code.
These tests compare it with arithmetic the oracle does not contain: the C
compiler's ``_Float16`` / ``__bf16`` casts, an exact binary64 sum rounded once,
numpy's float16 conversion and torch's bfloat16 conversion.
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


def run_pin(exe, test, lo=0, hi=0, stride=1):
    out = subprocess.run([exe, test, str(lo), str(hi), str(stride)], check=True,
                         capture_output=True, text=True).stdout.split()
    assert out[0] == test
    checked, bad, first = int(out[1]), int(out[2]), int(out[3])
    assert checked > 0
    assert bad == 0, f"{test}: {bad} mismatches of {checked}, first at input {first:#x}"
    return checked


def f32_exp_range(e_lo, e_hi):
    """Encodings of all binary32 values with biased exponent in [e_lo, e_hi], positive and negative."""
    return [(s + (e_lo << 23), s + ((e_hi + 1) << 23)) for s in (0, 1 << 31)]


def test_widening_exhaustive(pin_exe):
    assert run_pin(pin_exe, "f16_to_f32") == 65536
    assert run_pin(pin_exe, "bf16_to_f32") == 65536


def test_f32_to_f16_rounding(pin_exe):
    # every 7th binary32 encoding (7 is odd, so all low-bit patterns occur) ...
    run_pin(pin_exe, "f32_to_f16", 0, 1 << 32, 7)
    # ... plus every encoding in the subnormal range of binary16 and its edges
    # (|x| in [2^-26, 2^-13)), and around the overflow threshold (|x| in [2^14, 2^17))
    for lo, hi in f32_exp_range(101, 113) + f32_exp_range(141, 143):
        run_pin(pin_exe, "f32_to_f16", lo, hi)


def test_f32_to_bf16_rounding(pin_exe):
    run_pin(pin_exe, "f32_to_bf16", 0, 1 << 32, 3)
    # binary32 subnormals and the smallest normals, and the top of the range
    for lo, hi in f32_exp_range(0, 2) + f32_exp_range(253, 255):
        run_pin(pin_exe, "f32_to_bf16", lo, hi)


def test_hop_add_f16(pin_exe):
    # one hop = binary32 sum rounded once to binary16; checked against the exact
    # (binary64) sum rounded once, on every 13th pair of the 2^32 pairs ...
    run_pin(pin_exe, "add_f16", 0, 1 << 32, 13)
    # ... and on every pair whose first operand is a subnormal or a small normal
    run_pin(pin_exe, "add_f16", 0, 0x0800 << 16)
    run_pin(pin_exe, "add_f16", 0x8000 << 16, 0x8800 << 16)


def test_hop_add_bf16(pin_exe):
    run_pin(pin_exe, "add_bf16", 0, 1 << 32, 13)
    run_pin(pin_exe, "add_bf16", 0, 0x0100 << 16)
    run_pin(pin_exe, "add_bf16", 0x7f00 << 16, 0x7f80 << 16)


def test_hop_add_f32(pin_exe):
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
