"""The C ABI library loads, exports what include/k3moe.h declares, and refuses bad arguments
before touching a GPU (these tests need no GPU)."""
import ctypes
import re

import pytest

import mxfp4_routed_expert_06_b300 as k3


def _declared_functions():
    src = open(k3.HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(k3moe_\w+)\s*\(", src)))


def test_header_and_library_agree():
    declared = _declared_functions()
    assert declared == k3.exported_symbols()
    for name in declared:
        assert hasattr(k3._lib, name), name
        assert ctypes.cast(getattr(k3._lib, name), ctypes.c_void_p).value


def test_header_constants():
    assert k3.K3MOE_OK == 0
    assert k3.K3MOE_ERR_INVALID_ARG == -1 and k3.K3MOE_ERR_BUDGET_TOO_SMALL == -5
    assert k3.K3MOE_K_COUNT == len(k3.KERNEL_NAMES)


@pytest.mark.parametrize("dm,ok", [
    ((7168, 1536, 896, 16, 1), True),
    ((256, 128, 8, 2, 4), True),
    ((7168, 1536, 896, 33, 1), False),   # k > 32
    ((7168, 1500, 896, 16, 1), False),   # f not a multiple of 128
    ((100, 128, 8, 2, 4), False),        # d not a multiple of 128
    ((256, 128, 8, 9, 4), False),        # k > E
    ((256, 128, 0, 1, 4), False),
    ((256, 128, 8, 2, 0), False),
    ((256, 128, 8, 2, 70000), False),
])
def test_dims_validation(dm, ok):
    n = k3.k3moe_packed_expert_bytes(k3.dims(*dm))
    if ok:
        d, f = dm[0], dm[1]
        assert n == 3 * f * d // 2 + 3 * f * d // 32
    else:
        assert n == 0


def test_k3_packed_size_is_the_pages_count():
    assert k3.k3moe_packed_expert_bytes(k3.dims(7168, 1536, 896, 16, 1)) == 17_547_264


def test_bad_arguments_are_refused_without_device_work():
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_pack_experts(k3.dims(100, 128, 8, 2, 4), 1, 1, 1, 1)
    assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG and "d=100" in str(ei.value)
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_pack_experts(k3.dims(256, 128, 8, 2, 4), None, 1, 1, 1)
    assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_pack_experts(k3.dims(256, 128, 8, 2, 4), 1, 1, 2, 1)
    assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_cache_create(1000, 1024)
    assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_cache_create(1 << 30, 1000)
    assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG
    for fn, args in [(k3.k3moe_layer_forward, (None, 1, 1, 1)), (k3.k3moe_router_topk, (None, 1, 1, 1, 1)),
                     (k3.k3moe_bucket, (None, 1, 1, 1, 1, 1)), (k3.k3moe_set_option, (None, 1, 0)),
                     (k3.k3moe_profile, (None, 1)), (k3.k3moe_layer_set_cache, (None, 1)),
                     (k3.k3moe_residual_rmsnorm, (None, 16, 1, 8, 0.0, 32, 48)),
                     (k3.k3moe_residual_rmsnorm, (16, 32, 0, 8, 0.0, 48, 64)),
                     (k3.k3moe_residual_rmsnorm, (16, 32, 1, 70000, 0.0, 48, 64)),
                     (k3.k3moe_residual_rmsnorm, (16, 32, 1, 8, -1.0, 48, 64)),
                     (k3.k3moe_residual_rmsnorm, (16, 32, 1, 8, float("nan"), 48, 64)),
                     (k3.k3moe_residual_rmsnorm, (16, 32, 1, 8, 0.0, 48, 48))]:
        with pytest.raises(k3.K3MoEError) as ei:
            fn(*args)
        assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG


def test_free_null_is_harmless():
    k3.k3moe_layer_free(None)
    k3.k3moe_cache_destroy(None)


def _fnv1a64(b: bytes) -> int:
    x = 1469598103934665603
    for c in b:
        x = ((x ^ c) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return x


def _header(**kw):
    import ctypes
    h = k3.k3moe_pool_header(magic=k3.K3MOE_POOL_MAGIC, version=k3.K3MOE_POOL_VERSION, d=7168, f=1536, E=896,
                             s_min=121, s_max=125, zero_scales=0, expert_bytes=17547264)
    for k_, v in kw.items():
        setattr(h, k_, v)
    raw = bytes(h)[:k3.k3moe_pool_header.checksum.offset]
    h.checksum = _fnv1a64(raw)
    return h


def test_pool_header_check_accepts_a_valid_header_and_names_each_mismatch():
    dm = k3.dims(7168, 1536, 896, 16, 1)
    k3.k3moe_pool_header_check(_header(), dm)
    cases = [(dict(magic=0x12345678), "magic"), (dict(version=2), "version"), (dict(E=895), "E=895"),
             (dict(expert_bytes=17547263), "expert size"), (dict(s_min=126), "scale range"),
             (dict(s_min=0, zero_scales=0), "scale range"), (dict(s_max=255), "scale range")]
    for kw, needle in cases:
        with pytest.raises(k3.K3MoEError) as ei:
            k3.k3moe_pool_header_check(_header(**kw), dm)
        assert ei.value.code == k3.K3MOE_ERR_INVALID_ARG and needle in str(ei.value), (kw, str(ei.value))
    h = _header()
    h.s_max = 124  # changed after the checksum was taken
    with pytest.raises(k3.K3MoEError) as ei:
        k3.k3moe_pool_header_check(h, dm)
    assert "checksum" in str(ei.value)
    with pytest.raises(k3.K3MoEError):
        k3.k3moe_pool_header_check(_header(), k3.dims(7168, 1536, 896, 16, 0))  # invalid dims


def test_misaligned_buffers_are_refused_before_any_work():
    """Entry points that need no layer check their pointers' alignment before touching the device
    (these pointers are never dereferenced): a misaligned access would be a device fault."""
    cases = [
        # residual + RMSNorm: y float32, x / x_next / x_norm bf16
        lambda: k3._lib.k3moe_residual_rmsnorm(0x1002, 0x2000, 1, 8, 1e-6, 0x3000, 0x4000, None),
        lambda: k3._lib.k3moe_residual_rmsnorm(0x1000, 0x2001, 1, 8, 1e-6, 0x3000, 0x4000, None),
        lambda: k3._lib.k3moe_residual_rmsnorm(0x1000, 0x2000, 1, 8, 1e-6, 0x3001, 0x4000, None),
        # the no-alloc router: x 8-byte, W_r 16-byte, idx / w / bias 4-byte
        lambda: k3._lib.k3moe_router_topk_noalloc(0x1004, 0x2000, None, 1, 8, 4, 2, 0x3000, 0x4000, None),
        lambda: k3._lib.k3moe_router_topk_noalloc(0x1000, 0x2008, None, 1, 8, 4, 2, 0x3000, 0x4000, None),
        lambda: k3._lib.k3moe_router_topk_noalloc(0x1000, 0x2000, None, 1, 8, 4, 2, 0x3002, 0x4000, None),
        lambda: k3._lib.k3moe_router_topk_noalloc(0x1000, 0x2000, 0x5001, 1, 8, 4, 2, 0x3000, 0x4000, None),
    ]
    for i, call in enumerate(cases):
        assert call() == k3.K3MOE_ERR_INVALID_ARG, f"case {i}"
        assert "aligned" in k3._lib.k3moe_last_error().decode(), f"case {i}"
