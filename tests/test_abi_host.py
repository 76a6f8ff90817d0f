"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function ``include/moe_gb300.h`` declares,
and reject invalid layers on the host before touching CUDA.
"""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def nat():
    ensure_built()
    from routing_shared_expert_gb300 import _native
    return _native


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|moe_status)\s+(moe_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_grouped_swiglu", "moe_shared_mlp", "moe_combine",
              "moe_layer_forward", "moe_workspace_size", "moe_read_status"):
        assert n in names


def test_library_exports_every_declared_symbol(nat):
    lib = nat.library()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def _olmo(**kw):
    from workloads import CONFIGS
    from routing_shared_expert_gb300.layer import config_from_spec
    spec = CONFIGS["olmo"]
    c = config_from_spec(spec)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_workspace_size_valid_and_monotone(nat):
    a = nat.moe_workspace_size(_olmo(T=1024))
    b = nat.moe_workspace_size(_olmo(T=2048))
    assert 0 < a < b
    assert a % 256 == 0


@pytest.mark.parametrize("field,value,status", [
    ("K", 0, -1), ("K", 33, -1), ("N", 0, -1), ("N", 300, -1), ("T", -1, -1),
    ("dtype", 7, -1), ("score", 3, -1), ("norm", 9, -1), ("norm", 4, -1), ("shared_mode", 0, -1),
    ("cap_policy", 5, -1), ("num_ranks", 0, -1), ("alpha", float("nan"), -1),
    ("d_model", 100, -2), ("d_expert", 36, -2),
])
def test_invalid_layers_rejected_on_host(nat, field, value, status):
    c = _olmo(**{field: value})
    n = ctypes.c_size_t(0)
    got = nat.library().moe_workspace_size(ctypes.byref(c), ctypes.byref(n))
    assert got == status, (field, value, got)


def test_capacity_factor_checked_only_with_a_policy(nat):
    c = _olmo(capacity_factor=-1.0)
    assert nat.moe_workspace_size(c) > 0
    c = _olmo(capacity_factor=-1.0, cap_policy=1)
    with pytest.raises(nat.MoEError):
        nat.moe_workspace_size(c)


def test_lp_exponent_checked_only_with_the_lp_rule(nat):
    for p in (1.0, 2.0, 64.0):
        assert nat.moe_workspace_size(_olmo(norm=3, norm_p=p)) > 0
    for p in (0.5, 0.0, -2.0, 65.0, float("nan"), float("inf")):
        with pytest.raises(nat.MoEError):
            nat.moe_workspace_size(_olmo(norm=3, norm_p=p))
    # other rules ignore the field
    assert nat.moe_workspace_size(_olmo(norm=1, norm_p=float("nan"))) > 0


def test_backward_rejects_unsupported_layers(nat):
    # fp32 layers, and widths that are not multiples of 128
    with pytest.raises(nat.MoEError):
        nat.moe_backward_workspace_size(nat.make_config(T=16, d_model=64, N=8, K=2, d_expert=128,
                                                        d_shared=64, dtype="f32"))
    for kw in (dict(d_model=192), dict(d_expert=320), dict(d_shared=64)):
        c = _olmo(**kw)
        with pytest.raises(nat.MoEError) as e:
            nat.moe_backward_workspace_size(c)
        assert e.value.status == -2
    # the backward reads bf16 down projections: a layer configured for packed fp16 ones is
    # rejected, the same layer with the bf16 intermediate is accepted
    with pytest.raises(nat.MoEError) as e:
        nat.moe_backward_workspace_size(_olmo(h_format=1))
    assert e.value.status == -2
    assert nat.moe_backward_workspace_size(_olmo(h_format=0)) > nat.moe_workspace_size(_olmo())


def test_intermediate_format_fields_validated(nat):
    for kw in (dict(h_format=2), dict(h_format=-1), dict(h_scale_log2=65), dict(h_scale_log2=-65)):
        with pytest.raises(nat.MoEError) as e:
            nat.moe_workspace_size(_olmo(**kw))
        assert e.value.status == -1
    assert nat.moe_workspace_size(_olmo(h_format=1, h_scale_log2=-64)) > 0


def test_pack_weights_size_and_argument_checks(nat):
    import ctypes
    lib = nat.library()
    # a 256-byte header, then 2 bytes per element rounded up to 256 bytes
    assert nat.moe_packed_weights_size(0) == 256
    assert nat.moe_packed_weights_size(1) == 512
    assert nat.moe_packed_weights_size(128) == 512
    assert nat.moe_packed_weights_size(129) == 768
    n = ctypes.c_size_t(0)
    assert lib.moe_packed_weights_size(-1, ctypes.byref(n)) == -1
    assert lib.moe_packed_weights_size(8, None) == -1
    # null output, too small a buffer, misaligned pointers: rejected before anything is enqueued
    assert lib.moe_pack_weights(ctypes.c_void_p(4096), 64, None, 512, None) == -1
    assert lib.moe_pack_weights(ctypes.c_void_p(4096), 64, ctypes.c_void_p(1 << 20), 256, None) == -1
    assert lib.moe_pack_weights(None, 64, ctypes.c_void_p(1 << 20), 512, None) == -1
    assert lib.moe_pack_weights(ctypes.c_void_p(4096), 64, ctypes.c_void_p((1 << 20) + 16), 512,
                                None) == -7
    assert lib.moe_pack_weights(ctypes.c_void_p(4098), 64, ctypes.c_void_p(1 << 20), 512, None) == -7
    # overlapping input and output
    assert lib.moe_pack_weights(ctypes.c_void_p((1 << 20) + 256), 64, ctypes.c_void_p(1 << 20), 512,
                                None) == -1


def test_backward_rejects_null_arguments_before_cuda(nat):
    import ctypes
    lib = nat.library()
    c = _olmo(T=64, h_format=0)
    n = nat.moe_backward_workspace_size(c)
    assert n > 0
    w = nat.moe_weights()
    o = nat.moe_outputs()
    g = nat.moe_grads()
    # null weights / outputs / grads: invalid argument, nothing enqueued
    st = lib.moe_layer_backward(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(o), None,
                                ctypes.byref(g), None, 0, None)
    assert st == -1


def test_rho_out_of_range_rejected(nat):
    c = nat.make_config(T=16, d_model=64, N=4, K=1, d_expert=64, d_shared=0, shared_mode="none",
                        cap_policy="rank_wide", num_ranks=2, rho=[0, 1, 2, 0])
    with pytest.raises(nat.MoEError):
        nat.moe_workspace_size(c)


def test_entry_points_reject_before_cuda(nat):
    """Null workspace / null outputs are refused on the host; no CUDA call is made."""
    lib = nat.library()
    c = _olmo(T=64)
    fake = ctypes.c_void_p(0x1000)
    st = lib.moe_route(ctypes.byref(c), fake, fake, None, None, None, fake, fake, None, None, None,
                       0, None)
    assert st == -1
    st = lib.moe_route(ctypes.byref(c), fake, fake, None, None, None, fake, fake, None, None,
                       ctypes.c_void_p(0x100100), 16, None)
    assert st == -4   # workspace too small
    st = lib.moe_route(ctypes.byref(c), fake, fake, None, None, None, fake, fake, None, None,
                       ctypes.c_void_p(0x100101), 1 << 40, None)
    assert st == -7   # misaligned workspace
    w = nat.moe_weights()
    o = nat.moe_outputs()
    st = lib.moe_layer_forward(ctypes.byref(c), ctypes.byref(w), fake, ctypes.byref(o), None, 0, None)
    assert st == -1   # y missing
    # combine with g but no shared coefficient
    st = lib.moe_combine(ctypes.byref(c), fake, fake, fake, fake, None, fake, None)
    assert st == -1


def test_bias_update_and_stats_reject_bad_args(nat):
    lib = nat.library()
    fake = ctypes.c_void_p(0x1000)
    assert lib.moe_bias_update(0, fake, 0.1, fake, None) == -1
    assert lib.moe_bias_update(4, None, 0.1, fake, None) == -1
    assert lib.moe_bias_update(4, fake, float("inf"), fake, None) == -1
    c = _olmo(T=64)
    assert lib.moe_balance_stats(ctypes.byref(c), None, None, None, None, None, None, None, None,
                                 None, 0, None) == -1


def test_status_strings(nat):
    lib = nat.library()
    for code in range(-7, 1):
        assert lib.moe_status_string(code)
    assert nat.version().startswith("moe_gb300")


def test_wait_bound_check_rejects_before_cuda(nat):
    lib = nat.library()
    assert lib.moe_check_wait_bound(None, 1 << 20, 1000000, None) == -1          # no workspace
    assert lib.moe_check_wait_bound(ctypes.c_void_p(0x100000), 16, 1000000, None) == -1   # too small
    assert lib.moe_check_wait_bound(ctypes.c_void_p(0x100000), 1 << 20, 0, None) == -1    # no limit
    assert lib.moe_check_wait_bound(ctypes.c_void_p(0x100000), 1 << 20, 3000000000, None) == -1
    assert lib.moe_check_wait_bound(ctypes.c_void_p(0x100001), 1 << 20, 1000000, None) == -7  # misaligned
