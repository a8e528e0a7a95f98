"""The C-ABI library builds, loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (CPU only: no compute call reaches CUDA)."""

import ctypes
import os
import re
import subprocess

import pytest

import paged_gqa_attention_hd512_gb300 as pa
from paged_gqa_attention_hd512_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_attn.h")


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pa.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(paged_attn_\w+)\(", text, re.M)))


def test_header_declares_binding_names():
    assert declared_functions() == sorted(pa.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (paged_attn_\w+)", out))
    assert set(declared_functions()) <= exported
    for name in declared_functions():
        assert hasattr(lib, name)


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5, -6, -7):
        assert pa.paged_attn_status_string(st)
    assert pa.paged_attn_status_string(-99) == "unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation rejects before any CUDA call


def _decode(lib, **over):
    a = dict(q=FAKE, kv=FAKE, ip=FAKE, ind=FAKE, last=FAKE, batch=2, num_pages=4, hq=8, hkv=1,
             dqk=512, dvo=512, ps=16, scale=0.04, win=-1, dt=0, out=FAKE, lse=None)
    a.update(over)
    sc = pa._Scales(None, None, None)
    return lib.paged_attn_decode(a["q"], a["kv"], a["ip"], a["ind"], a["last"], a["batch"], a["num_pages"],
                                 a["hq"], a["hkv"], a["dqk"], a["dvo"], a["ps"], a["scale"], a["win"],
                                 a["dt"], ctypes.byref(sc), a["out"], a["lse"], None)


def test_decode_rejects_bad_arguments(lib):
    assert _decode(lib, q=None) == pa.PA_ERR_INVALID_ARG
    assert _decode(lib, hq=7, hkv=2) == pa.PA_ERR_INVALID_ARG
    assert _decode(lib, hq=34, hkv=2) == pa.PA_ERR_UNSUPPORTED  # group 17
    assert _decode(lib, dqk=384, dvo=384) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, dqk=256, dvo=512) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, ps=12) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, ps=128) == pa.PA_ERR_UNSUPPORTED
    assert _decode(lib, q=FAKE + 8) == pa.PA_ERR_ALIGNMENT
    assert _decode(lib, win=-2) == pa.PA_ERR_INVALID_ARG
    assert _decode(lib, dt=1) == pa.PA_ERR_INVALID_ARG  # FP8 without scales
    assert _decode(lib, dt=7) == pa.PA_ERR_INVALID_ARG
    assert _decode(lib, num_pages=0) == pa.PA_ERR_INVALID_ARG
    assert _decode(lib, scale=float("nan")) == pa.PA_ERR_INVALID_ARG


def test_prefill_rejects_bad_arguments(lib):
    sc = pa._Scales(None, None, None)
    st = lib.paged_attn_prefill(FAKE, None, 10, FAKE, FAKE, FAKE, FAKE, 1, 4, 8, 1, 512, 512, 16, 0.04, -1, 1,
                                0, ctypes.byref(sc), FAKE, None, None)
    assert st == pa.PA_ERR_INVALID_ARG
    st = lib.paged_attn_prefill(FAKE, FAKE, 10, FAKE, FAKE, FAKE, FAKE, 1, 4, 8, 3, 512, 512, 16, 0.04, -1, 1,
                                0, ctypes.byref(sc), FAKE, None, None)
    assert st == pa.PA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 8, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.paged_attn_decode(q, torch.zeros(10, dtype=torch.uint8), torch.zeros(2, dtype=torch.int32),
                             torch.zeros(1, dtype=torch.int32), torch.ones(1, dtype=torch.int32),
                             num_kv_heads=1, head_dim_vo=512, page_size=16, sm_scale=0.04, num_pages=1)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        pa.load(str(tmp_path / "nope.so"))


def test_prefill_custom_mask_rejects_bad_arguments(lib):
    sc = pa._Scales(None, None, None)
    args = (FAKE, FAKE, 10, FAKE, FAKE, FAKE, FAKE, 1, 4, 8, 1, 512, 512, 16, 0.04, -1, 1, 0, ctypes.byref(sc),
            FAKE, None)
    assert lib.paged_attn_prefill_custom_mask(*args, None, FAKE, None) == pa.PA_ERR_INVALID_ARG
    assert lib.paged_attn_prefill_custom_mask(*args, FAKE, None, None) == pa.PA_ERR_INVALID_ARG
    assert lib.paged_attn_prefill_custom_mask(*args, FAKE, FAKE + 4, None) == pa.PA_ERR_ALIGNMENT


def _append(lib, **over):
    a = dict(k=FAKE, v=FAKE, ai=FAKE, total=8, cache=FAKE, ip=FAKE, ind=FAKE, last=FAKE, batch=2, num_pages=4,
             hkv=2, dqk=512, dvo=256, ps=16, dt=0, ks=None, vs=None, sf=None)
    a.update(over)
    return lib.paged_attn_append_kv(a["k"], a["v"], a["ai"], a["total"], a["cache"], a["ip"], a["ind"], a["last"],
                                    a["batch"], a["num_pages"], a["hkv"], a["dqk"], a["dvo"], a["ps"], a["dt"],
                                    a["ks"], a["vs"], a["sf"], None)


def test_append_rejects_bad_arguments(lib):
    assert _append(lib, batch=0) == pa.PA_OK and _append(lib, total=0) == pa.PA_OK  # nothing to write
    assert _append(lib, k=None) == pa.PA_ERR_INVALID_ARG
    assert _append(lib, ai=None) == pa.PA_ERR_INVALID_ARG
    assert _append(lib, total=-1) == pa.PA_ERR_INVALID_ARG
    assert _append(lib, num_pages=0) == pa.PA_ERR_INVALID_ARG
    assert _append(lib, dqk=256, dvo=512) == pa.PA_ERR_UNSUPPORTED
    assert _append(lib, ps=24) == pa.PA_ERR_UNSUPPORTED
    assert _append(lib, dt=5) == pa.PA_ERR_INVALID_ARG
    assert _append(lib, dt=1) == pa.PA_ERR_INVALID_ARG  # FP8 without scales
    assert _append(lib, dt=2, ks=FAKE, vs=FAKE) == pa.PA_ERR_INVALID_ARG  # NVFP4 without a scale pool
    assert _append(lib, dt=1, ks=FAKE + 2, vs=FAKE) == pa.PA_ERR_ALIGNMENT
    assert _append(lib, k=FAKE + 8) == pa.PA_ERR_ALIGNMENT
    assert _append(lib, cache=FAKE + 8) == pa.PA_ERR_ALIGNMENT
    # one page of 2^14 kv heads x 64 rows x 2048 bytes of bf16 K and V: 2^31 bytes
    assert _append(lib, hkv=1 << 14, ps=64, dqk=512, dvo=512) == pa.PA_ERR_UNSUPPORTED


def test_mode_setters_reject_other_values(lib):
    assert lib.paged_attn_set_prefill_cta_pairs(2) == pa.PA_ERR_INVALID_ARG
    assert lib.paged_attn_set_prefill_split_kv(1) == pa.PA_ERR_INVALID_ARG
    assert lib.paged_attn_set_prefill_cta_pairs(-1) == pa.PA_OK
    assert lib.paged_attn_set_prefill_split_kv(-1) == pa.PA_OK
    for bad in (2, -2):
        assert lib.paged_attn_set_decode_direct(bad) == pa.PA_ERR_INVALID_ARG
    for ok in (0, 1, -1):
        assert lib.paged_attn_set_decode_direct(ok) == pa.PA_OK


def _decode_noalloc(lib, **over):
    a = dict(q=FAKE, kv=FAKE, ip=FAKE, ind=FAKE, last=FAKE, batch=2, num_pages=4, hq=8, hkv=1,
             dqk=512, dvo=512, ps=16, scale=0.04, win=-1, dt=0, out=FAKE, lse=None)
    a.update(over)
    sc = pa._Scales(None, None, None)
    return lib.paged_attn_decode_noalloc(a["q"], a["kv"], a["ip"], a["ind"], a["last"], a["batch"],
                                         a["num_pages"], a["hq"], a["hkv"], a["dqk"], a["dvo"], a["ps"],
                                         a["scale"], a["win"], a["dt"], ctypes.byref(sc), a["out"], a["lse"], None)


def test_decode_noalloc_rejects_bad_arguments(lib):
    assert _decode_noalloc(lib, batch=0) == pa.PA_OK  # nothing to do
    assert _decode_noalloc(lib, q=None) == pa.PA_ERR_INVALID_ARG
    assert _decode_noalloc(lib, out=None) == pa.PA_ERR_INVALID_ARG
    assert _decode_noalloc(lib, kv=None) == pa.PA_ERR_INVALID_ARG
    assert _decode_noalloc(lib, hq=7, hkv=2) == pa.PA_ERR_INVALID_ARG
    assert _decode_noalloc(lib, hq=34, hkv=2) == pa.PA_ERR_UNSUPPORTED  # group 17
    assert _decode_noalloc(lib, ps=3) == pa.PA_ERR_UNSUPPORTED
    assert _decode_noalloc(lib, q=FAKE + 8) == pa.PA_ERR_ALIGNMENT
    assert _decode_noalloc(lib, out=FAKE + 4) == pa.PA_ERR_ALIGNMENT
    assert _decode_noalloc(lib, lse=FAKE + 2) == pa.PA_ERR_ALIGNMENT
    assert _decode_noalloc(lib, dt=2) == pa.PA_ERR_INVALID_ARG  # NVFP4 without scales
    assert _decode_noalloc(lib, win=-3) == pa.PA_ERR_INVALID_ARG


def test_debug_error_hook_rejects_unknown_target(lib):
    assert lib.paged_attn_debug_set_error_word(2, 5) == pa.PA_ERR_INVALID_ARG
    assert lib.paged_attn_debug_set_error_word(-1, 5) == pa.PA_ERR_INVALID_ARG
