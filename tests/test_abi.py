"""The C-ABI library loads and exports every function include/gdn.h declares,
and its host-side argument checks answer without touching a GPU (CPU)."""
import os
import re

import pytest

import gated_deltanet_recurrence_gdn_gb300 as gdn
from gated_deltanet_recurrence_gdn_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gdn.load()


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("gdn_fwd", "gdn_fwd_varlen", "gdn_status_string", "gdn_sync_check"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the binding declares a prototype for each of them
    bound = {n for n, _, _ in gdn.ABI}
    assert set(declared_functions()) <= bound


def test_status_strings(lib):
    for s in range(8):
        assert lib.gdn_status_string(s).decode().startswith("GDN_")
    assert lib.gdn_status_string(99) == b"unknown gdn_status"


def test_options_roundtrip(lib):
    assert lib.gdn_set_option(gdn.GDN_OPT_IMPL, gdn.GDN_IMPL_SIMT) == gdn.GDN_OK
    assert lib.gdn_get_option(gdn.GDN_OPT_IMPL) == gdn.GDN_IMPL_SIMT
    assert lib.gdn_set_option(gdn.GDN_OPT_IMPL, 9) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_set_option(77, 0) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_set_option(gdn.GDN_OPT_IMPL, gdn.GDN_IMPL_AUTO) == gdn.GDN_OK
    prev = lib.gdn_get_option(gdn.GDN_OPT_POISON_SCRATCH)
    assert lib.gdn_set_option(gdn.GDN_OPT_POISON_SCRATCH, 1) == gdn.GDN_OK
    assert lib.gdn_get_option(gdn.GDN_OPT_POISON_SCRATCH) == 1
    assert lib.gdn_set_option(gdn.GDN_OPT_POISON_SCRATCH, 2) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_set_option(gdn.GDN_OPT_POISON_SCRATCH, prev) == gdn.GDN_OK
    prev = lib.gdn_get_option(gdn.GDN_OPT_HOST_SLICE)
    assert lib.gdn_set_option(gdn.GDN_OPT_HOST_SLICE, 1024) == gdn.GDN_OK
    assert lib.gdn_get_option(gdn.GDN_OPT_HOST_SLICE) == 1024
    assert lib.gdn_set_option(gdn.GDN_OPT_HOST_SLICE, -1) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_set_option(gdn.GDN_OPT_HOST_SLICE, prev) == gdn.GDN_OK
    prev = lib.gdn_get_option(gdn.GDN_OPT_PREP_LEAD)
    assert prev == 0   # automatic by default
    for v in (-1, 1, 48):
        assert lib.gdn_set_option(gdn.GDN_OPT_PREP_LEAD, v) == gdn.GDN_OK
        assert lib.gdn_get_option(gdn.GDN_OPT_PREP_LEAD) == v
    assert lib.gdn_set_option(gdn.GDN_OPT_PREP_LEAD, -2) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_set_option(gdn.GDN_OPT_PREP_LEAD, prev) == gdn.GDN_OK


# Host-only validation: these calls must return before any CUDA call, so fake
# (never dereferenced) device addresses are fine.
FAKE = 0x10000


def _args(off=0):
    return [FAKE + off, FAKE, FAKE, FAKE, FAKE, None, FAKE, None]


def test_host_checks(lib):
    f = lib.gdn_fwd
    assert f(*_args(), 1, 1, 64, 64, 64, 128, 1, None) == gdn.GDN_ERR_UNSUPPORTED  # chunk
    assert f(*_args(), 1, 1, 64, 60, 64, 64, 1, None) == gdn.GDN_ERR_UNSUPPORTED   # d_k % 8
    assert f(*_args(), 1, 1, 64, 256, 64, 64, 1, None) == gdn.GDN_ERR_UNSUPPORTED  # d_k > 128
    assert f(*_args(), 1, 1, 64, 64, 512, 64, 1, None) == gdn.GDN_ERR_UNSUPPORTED  # d_v > 256
    assert f(*_args(8), 1, 1, 64, 64, 64, 64, 1, None) == gdn.GDN_ERR_ALIGNMENT
    assert f(*_args(), -1, 1, 64, 64, 64, 64, 1, None) == gdn.GDN_ERR_INVALID_ARG
    assert f(*_args(), 1, 1, 64, 64, 64, 64, 3, None) == gdn.GDN_ERR_INVALID_ARG   # dtype
    nul = _args()
    nul[2] = None
    assert f(*nul, 1, 1, 64, 64, 64, 64, 1, None) == gdn.GDN_ERR_INVALID_ARG
    # nothing to do: zero heads / zero batch returns OK without launching
    assert f(*_args(), 0, 4, 64, 64, 64, 64, 1, None) == gdn.GDN_OK
    assert f(*_args(), 2, 0, 64, 64, 64, 64, 1, None) == gdn.GDN_OK
    g = lib.gdn_fwd_varlen
    assert g(*_args(), None, 2, 1, 10, 64, 64, 64, 1, None) == gdn.GDN_ERR_INVALID_ARG
    assert g(*_args(), FAKE, 0, 1, 10, 64, 64, 64, 1, None) == gdn.GDN_ERR_INVALID_ARG
    assert g(*_args(), FAKE, 0, 1, 0, 64, 64, 64, 1, None) == gdn.GDN_OK
    # variant flags: both known bits pass the checks, any other bit is refused
    fx, gx = lib.gdn_fwd_ex, lib.gdn_fwd_varlen_ex
    both = gdn.GDN_FLAG_NO_ERASE | gdn.GDN_FLAG_VECTOR_GATE
    assert fx(*_args(), 0, 4, 64, 64, 64, 64, 1, both, None) == gdn.GDN_OK
    assert fx(*_args(), 0, 4, 64, 64, 64, 64, 1, 4, None) == gdn.GDN_ERR_INVALID_ARG
    assert gx(*_args(), FAKE, 0, 1, 0, 64, 64, 64, 1, both, None) == gdn.GDN_OK
    assert gx(*_args(), FAKE, 0, 1, 0, 64, 64, 64, 1, 8, None) == gdn.GDN_ERR_INVALID_ARG


def test_bwd_host_checks(lib):
    f = lib.gdn_bwd
    a = [FAKE] * 14
    assert f(*a, 0, 2, 64, 64, 64, 64, 1, 0, None) == gdn.GDN_OK                 # nothing to do
    assert f(*a, 0, 2, 64, 64, 64, 64, 1, 4, None) == gdn.GDN_ERR_INVALID_ARG    # flag bit
    assert f(*a, 0, 2, 64, 64, 64, 64, 1, gdn.GDN_FLAG_VECTOR_GATE, None) == \
        gdn.GDN_ERR_UNSUPPORTED
    assert f(*a, 1, 1, 64, 64, 64, 128, 1, 0, None) == gdn.GDN_ERR_UNSUPPORTED   # chunk
    nul = list(a)
    nul[8] = None                                                                # dq
    assert f(*nul, 1, 1, 64, 64, 64, 64, 1, 0, None) == gdn.GDN_ERR_INVALID_ARG
    mis = list(a)
    mis[11] = FAKE + 4                                                           # dlog_alpha
    assert f(*mis, 1, 1, 64, 64, 64, 64, 1, 0, None) == gdn.GDN_ERR_ALIGNMENT
    g = lib.gdn_bwd_varlen
    assert g(*a, None, 2, 1, 10, 64, 64, 64, 1, 0, None) == gdn.GDN_ERR_INVALID_ARG
    assert g(*a, FAKE, 0, 1, 0, 64, 64, 64, 1, 0, None) == gdn.GDN_OK


def test_decode_host_checks(lib):
    f = lib.gdn_decode
    a = [FAKE] * 6 + [None, 0, FAKE]
    assert f(*a, 2, 2, 48, 64, 1, None) == gdn.GDN_ERR_UNSUPPORTED    # d_k
    assert f(*a, 2, 2, 64, 0, 1, None) == gdn.GDN_ERR_INVALID_ARG     # d_v
    assert f(*a, 2, 2, 64, 64, 3, None) == gdn.GDN_ERR_INVALID_ARG    # dtype
    assert f(*a, -1, 2, 64, 64, 1, None) == gdn.GDN_ERR_INVALID_ARG   # B
    assert f(*a, 0, 2, 64, 64, 1, None) == gdn.GDN_OK                 # nothing to do
    slots = [FAKE] * 6 + [FAKE, 0, FAKE]
    assert f(*slots, 2, 2, 64, 64, 1, None) == gdn.GDN_ERR_INVALID_ARG  # empty pool
    mis = list(a)
    mis[5] = FAKE + 8
    assert f(*mis, 2, 2, 64, 64, 1, None) == gdn.GDN_ERR_ALIGNMENT


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        gdn.load(str(tmp_path / "missing.so"))


def test_selftest_argument_checks(lib):
    # rejected on the host, before any CUDA call
    for complete, limit in ((2, 10), (-1, 10), (0, 0), (1, -5), (0, (1 << 22) + 1)):
        assert lib.gdn_selftest_wait(complete, limit, None, None) == gdn.GDN_ERR_INVALID_ARG


def test_build_targets_sm103a_only():
    flags = _build.ARCH
    assert flags == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_binding_refuses_host_tensors(lib):
    # no CPU fallback: host tensors are rejected before anything runs
    import torch
    x = torch.zeros(1, 1, 4, 8)
    g = torch.zeros(1, 1, 4)
    with pytest.raises(ValueError):
        gdn.gdn_fwd(x, x, x, g, g)
    with pytest.raises(ValueError):
        gdn.gdn_decode(x[:, :, 0], x[:, :, 0], x[:, :, 0], g[:, :, 0], g[:, :, 0],
                       torch.zeros(1, 1, 8, 8))
