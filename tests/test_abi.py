"""The C-ABI library loads and exports every entry point its header declares;
host-only entry points (layout, status strings, argument checks) behave as
documented.  No GPU needed: nothing here launches work."""
import ctypes
import os
import re

import pytest

import oracle
from continuous_linear_attention_gb300 import binding

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")


def _declared(headers=("gdn.h", "gdn_diag.h")):
    src = "".join(open(os.path.join(INCLUDE, h)).read() for h in headers)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    lib = binding.load()
    names = _declared()
    assert "gdn_varlen_forward" in names and "gdn_state_pool_create" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(binding.EXPORTED + ["gdn_diag_umma_gemm", "gdn_diag_umma_gemm_ex",
                                      "gdn_diag_wait_timeout"]) == names
    assert "gdn_kda_varlen_forward" in names and "gdn_ssd_varlen_forward" in names


@pytest.mark.parametrize("dims", [
    (512, 1, 16, 32, 128, 128, 4, "bf16", 0),
    (8, 1, 2, 4, 32, 32, 4, "f32", 0),
    (1024, 3, 16, 32, 128, 128, 4, "bf16", 4096),
    (4, 2, 1, 1, 64, 64, 2, "bf16", 0),
    (4, 2, 2, 2, 32, 32, 3, "bf16", 1 << 16),
])
def test_layout_matches_the_stated_layout(dims):
    nb, nl, Hk, Hv, dk, dv, K, act, align = dims
    stride, conv_off, rec_off, total = binding.layout_for(nb, nl, Hk, Hv, dk, dv, K, act, align)
    spec = oracle.pool_layout(nb, nl, Hk, Hv, dk, dv, K, 4 if act == "f32" else 2, align)
    assert (stride, conv_off, rec_off, total) == (spec["stride"], spec["conv_off"],
                                                  spec["rec_off"], spec["total"])
    assert rec_off % 128 == 0 and stride % 128 == 0


@pytest.mark.parametrize("bad", [
    dict(dk=48, dv=48), dict(dk=64, dv=128), dict(Hv=3), dict(Hv=64), dict(K=1), dict(K=5),
    dict(align=100), dict(align=64),
])
def test_layout_rejects_unsupported_dims(bad):
    args = dict(nb=8, nl=1, Hk=2, Hv=4, dk=32, dv=32, K=4, act="f32", align=0)
    args.update(bad)
    with pytest.raises(binding.GdnError) as e:
        binding.layout_for(args["nb"], args["nl"], args["Hk"], args["Hv"], args["dk"], args["dv"],
                           args["K"], args["act"], args["align"])
    assert e.value.status == -2


def test_layout_rejects_small_pools():
    with pytest.raises(binding.GdnError) as e:
        binding.layout_for(1, 1, 2, 4, 32, 32, 4, "f32", 0)
    assert e.value.status == -3


def test_status_strings():
    for code in range(-7, 1):
        assert binding.status_string(code) != "unknown status"
    assert binding.status_string(-99) == "unknown status"


def test_null_arguments_are_rejected_without_device_work():
    lib = binding.load()
    assert lib.gdn_state_pool_create(None, 8, 1, 2, 4, 32, 32, 4, 0, 0, None, 0) == -1
    w = binding.Weights(None, None, None)
    assert lib.gdn_varlen_forward(None, 0, None, None, None, None, None, None, ctypes.byref(w),
                                  None, 0, 0, 0, None) == -1
    v = ctypes.c_uint32()
    assert lib.gdn_get_error(None, 0, ctypes.byref(v), 0, None) == -1
    assert lib.gdn_kda_varlen_forward(None, 0, None, None, None, None, None, None,
                                      ctypes.byref(w), None, 0, 0, 0, None) == -1
    assert lib.gdn_state_pool_destroy(None) == 0
    assert lib.gdn_state_pool_layout(None, None, None, None, None) == -1


def test_wait_timeout_arguments_are_checked_on_the_host():
    lib = binding.load()
    buf = (ctypes.c_uint32 * 2)()
    assert lib.gdn_diag_wait_timeout(None, None) == -1
    misaligned = ctypes.c_void_p(ctypes.addressof(buf) + 2)
    assert lib.gdn_diag_wait_timeout(misaligned, None) == -4


@pytest.mark.parametrize("dims", [
    (512, 1, 128, 64, 128, 8, 4, "bf16", 0),
    (8, 1, 4, 32, 32, 2, 4, "f32", 0),
    (16, 3, 8, 64, 64, 1, 3, "bf16", 4096),
    (4, 2, 2, 32, 128, 2, 2, "f32", 1 << 16),
])
def test_ssd_layout_matches_the_stated_layout(dims):
    nb, nl, H, P, N, G, K, act, align = dims
    stride, conv_off, ssm_off, total = binding.ssd_layout_for(nb, nl, H, P, N, G, K, act, align)
    spec = oracle.ssd_pool_layout(nb, nl, H, P, N, G, K, 4 if act == "f32" else 2, align)
    assert (stride, conv_off, ssm_off, total) == (spec["stride"], spec["conv_off"],
                                                  spec["ssm_off"], spec["total"])
    assert ssm_off % 128 == 0 and stride % 128 == 0


@pytest.mark.parametrize("bad", [
    dict(P=16), dict(P=128), dict(N=16), dict(N=256), dict(G=3), dict(H=6, G=4), dict(K=1),
    dict(K=5), dict(align=100),
])
def test_ssd_layout_rejects_unsupported_dims(bad):
    args = dict(nb=8, nl=1, H=4, P=32, N=32, G=2, K=4, act="f32", align=0)
    args.update(bad)
    with pytest.raises(binding.GdnError) as e:
        binding.ssd_layout_for(args["nb"], args["nl"], args["H"], args["P"], args["N"], args["G"],
                               args["K"], args["act"], args["align"])
    assert e.value.status == -2


def test_ssd_null_arguments_are_rejected_without_device_work():
    lib = binding.load()
    assert lib.gdn_ssd_pool_create(None, 8, 1, 4, 32, 32, 2, 4, 0, 0, None, 0) == -1
    w = binding.SsdWeights(None, None, None, None)
    assert lib.gdn_ssd_varlen_forward(None, 0, None, None, None, None, None, ctypes.byref(w),
                                      None, 0, 0, 0, None) == -1


def test_prefill_scratch_bytes_grows_with_the_call():
    """The scratch size query: one slot per 64-token chunk plus one per
    possible prefill sequence, and argument checks."""
    small = binding.prefill_scratch_bytes(64, 16, 32, 128, 128, 64)
    large = binding.prefill_scratch_bytes(64, 16, 32, 128, 128, 16384)
    assert 0 < small < large
    with pytest.raises(binding.GdnError):
        binding.prefill_scratch_bytes(1, 16, 32, 128, 128, 64)
