"""The C ABI without a GPU: the library builds and loads, exports every
symbol the header declares, the header is plain C, and host-side argument
checks and planning answer without touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

import grouped_query_kv_gb300 as g
from grouped_query_kv_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvattn.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return g.lib()


def header_symbols():
    text = open(HEADER).read()
    names = re.findall(r"^KVATTN_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_binding_signatures():
    assert header_symbols() == sorted(g.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", g.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    for name in header_symbols():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_header_is_plain_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "kvattn.h"\nint main(void){kvattn_plan p; (void)p; '
                   'return (int)KVATTN_OK;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only",
                    "-I", os.path.dirname(HEADER), str(src)], check=True)


def test_status_strings(lib):
    assert lib.kvattn_status_string(0) == b"KVATTN_OK"
    assert lib.kvattn_status_string(5) == b"KVATTN_ERR_DEVICE_BOUNDS"
    assert lib.kvattn_status_string(99) == b"KVATTN_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: checks fail first


@pytest.mark.parametrize("args,status", [
    # null pointer
    ((None, FAKE, FAKE, FAKE, FAKE, 2, 4, 1, 64, 64, 0.1), g.KVATTN_ERR_INVALID_ARG),
    # misaligned
    ((ctypes.c_void_p(0x10002), FAKE, FAKE, FAKE, FAKE, 2, 4, 1, 64, 64, 0.1),
     g.KVATTN_ERR_INVALID_ARG),
    # Hq not a multiple of Hkv
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 6, 4, 64, 64, 0.1), g.KVATTN_ERR_INVALID_ARG),
    # non-positive sizes
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 1, 64, 64, 0.1), g.KVATTN_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 1, 64, 0, 0.1), g.KVATTN_ERR_INVALID_ARG),
    # unsupported head dim
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 1, 96, 64, 0.1), g.KVATTN_ERR_UNSUPPORTED),
    # non-finite scale
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 1, 64, 64, float("nan")), g.KVATTN_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 1, 64, 64, float("inf")), g.KVATTN_ERR_INVALID_ARG),
    # beyond limits
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 70000, 4, 1, 64, 64, 0.1), g.KVATTN_ERR_UNSUPPORTED),
])
def test_attention_argument_checks(lib, args, status):
    q, k, v, lens, out, B, Hq, Hkv, D, Lmax, scale = args
    rc = lib.gqa_decode_attn(q, k, v, lens, out, B, Hq, Hkv, D, Lmax, scale, None)
    assert rc == status
    assert lib.kvattn_last_error().decode() != ""


@pytest.mark.parametrize("args,status", [
    ((None, FAKE, FAKE, FAKE, FAKE, 2, 1, 64, 64), g.KVATTN_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, ctypes.c_void_p(0x10008), FAKE, 2, 1, 64, 64), g.KVATTN_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, 1, 32, 64), g.KVATTN_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 2, -1, 64, 64), g.KVATTN_ERR_INVALID_ARG),
])
def test_append_argument_checks(lib, args, status):
    rc = lib.kv_append(*args, None)
    assert rc == status


def test_tuning_knob_range(lib):
    assert lib.kvattn_set_tuning(3, 0) == g.KVATTN_ERR_INVALID_ARG
    assert lib.kvattn_set_tuning(0, -1) == g.KVATTN_ERR_INVALID_ARG
    assert lib.kvattn_set_tuning(0, 0) == g.KVATTN_OK


@pytest.mark.parametrize("B,Hq,Hkv,D,Lmax", [
    (2, 4, 1, 64, 64), (64, 16, 1, 256, 2048), (32, 64, 8, 128, 8192),
    (8, 48, 1, 256, 32768), (256, 32, 32, 128, 4096), (1, 32, 1, 128, 4096),
])
def test_plan_is_host_only_and_sane(lib, B, Hq, Hkv, D, Lmax):
    p = g.get_plan(B, Hq, Hkv, D, Lmax, num_sms=152)
    G = Hq // Hkv
    assert p["path"] in (1, 2)
    assert p["heads_per_cta"] * p["head_groups"] >= G
    assert (p["head_groups"] - 1) * p["heads_per_cta"] < G
    assert p["tile_positions"] in (64, 128, 256)
    assert p["num_ctas"] >= 1 and p["num_ctas"] % 152 == 0
    assert p["smem_bytes"] <= 232448  # 227 KB opt-in limit per CTA
    assert p["workspace_bytes"] >= 2 * p["num_ctas"] * p["heads_per_cta"] * (D + 2) * 4


def test_plan_honours_forced_grid(lib):
    g.set_tuning(0, 7)
    try:
        assert g.get_plan(8, 48, 1, 256, 32768, num_sms=152)["num_ctas"] == 7
    finally:
        g.set_tuning(0, 0)
