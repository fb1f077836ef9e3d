"""The C ABI without a GPU: the library loads, exports what include/moe.h declares,
and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

import oracle
import sparse_mixture_experts_62_b300 as moe

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MOE_API\s+[^(]*?\b(moe_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(moe.LIB_PATH)
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.EXPORTS)


def test_status_strings():
    for c in range(7):
        assert moe.status_string(c) and moe.status_string(c) != "unknown status"
    assert moe.status_string(99) == "unknown status"


@pytest.mark.parametrize("alpha,T,k,N", [(1.25, 16384, 8, 128), (1.0, 10, 2, 3), (1.1, 10, 1, 1), (0.5, 3, 1, 2),
                                         (2.0, 4096, 2, 8), (4.0, 16, 2, 8), (1.0, 0, 2, 8), (0.3, 777, 3, 7),
                                         (1.0 / 3.0, 3, 1, 1), (1e-3, 1, 1, 1)])
def test_capacity_matches_oracle(alpha, T, k, N):
    assert moe.moe_capacity(alpha, T, k, N) == oracle.capacity(alpha, T, k, N)


def test_capacity_rejects_bad_args():
    for args in [(0.0, 1, 1, 1), (-1.0, 1, 1, 1), (1.0, -1, 1, 1), (1.0, 1, 0, 1), (1.0, 1, 1, 0)]:
        with pytest.raises(moe.MoeError) as e:
            moe.moe_capacity(*args)
        assert e.value.code == moe.MOE_ERR_INVALID_ARG


def test_workspace_layout_is_aligned_and_sized():
    cfg = moe.make_config(8192, 7168, 256, 8, 2048, 2048, gate=moe.GATE_SIGMOID_BIAS)
    L = moe.moe_workspace_layout(cfg)
    fields = [f for f, _ in moe.MoeWsLayout._fields_]
    offs = [getattr(L, f) for f in fields]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.x_perm - L.src_token >= 8192 * 8 * 4
    assert L.h - L.x_perm >= 8192 * 8 * 7168 * 2
    assert L.total == moe.moe_workspace_size(cfg)


BAD_CONFIGS = [
    (dict(N=300), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=9, N=16), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=5, N=4), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=12), moe.MOE_ERR_UNSUPPORTED),        # bf16 rows must be 16-byte multiples
    (dict(ffn=100), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(N=0), moe.MOE_ERR_INVALID_ARG),
    (dict(gate=7), moe.MOE_ERR_INVALID_ARG),
    (dict(act=3), moe.MOE_ERR_INVALID_ARG),
    (dict(dtype=5), moe.MOE_ERR_INVALID_ARG),
    (dict(routing=2), moe.MOE_ERR_INVALID_ARG),
    (dict(routing=1, capacity=0), moe.MOE_ERR_INVALID_ARG),   # expert choice needs C >= 1
]


@pytest.mark.parametrize("kw,code", BAD_CONFIGS)
def test_bad_configs_rejected(kw, code):
    base = dict(T=64, d=64, N=8, k=2, ffn=128, shared_ffn=0, gate=0, act=1, dtype=1, capacity=0, routing=0)
    base.update(kw)
    cfg = moe.MoeConfig(*[base[f] for f, _ in moe.MoeConfig._fields_])
    with pytest.raises(moe.MoeError) as e:
        moe.moe_workspace_size(cfg)
    assert e.value.code == code
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_forward(cfg, 16, 16, None, None, 16, 16, 16, None, None, None, 16, 256, 0)
    assert e.value.code == code


def test_null_and_misaligned_pointers_rejected_without_launch():
    cfg = moe.make_config(64, 64, 8, 2, 128)
    A = 1 << 20  # a 256-aligned fake address: never dereferenced, validation fails first
    cases = [
        lambda: moe.moe_route(cfg, None, A, None, None, A, A, A, A, 0),
        lambda: moe.moe_route(cfg, A + 8, A, None, None, A, A, A, A, 0),          # x misaligned
        lambda: moe.moe_route(cfg, A, A, None, None, A, A, A, A + 16, 0),         # ws not 256-aligned
        lambda: moe.moe_expert_ffn(cfg, A, A, A, None, A, A, A, 0),               # swiglu needs w3
        lambda: moe.moe_combine(cfg, A, None, A, None, A, 0),
        lambda: moe.moe_shared_ffn(cfg, A, A, A, A, A, A, 0),                     # no shared expert in cfg
        lambda: moe.moe_layer_forward(cfg, A, A, None, None, A, A, A, None, None, None, A, None, 0),
        lambda: moe.moe_load_stats(cfg, None, A, A, A, A, A, A, 0),
        lambda: moe.moe_get_device_status(None, 0),
    ]
    for fn in cases:
        with pytest.raises(moe.MoeError) as e:
            fn()
        assert e.value.code == moe.MOE_ERR_INVALID_ARG


def test_fp8_entry_points_reject_bad_arguments_without_launch():
    A = 1 << 20
    cfg = moe.make_config(64, 64, 8, 2, 128)
    invalid = [
        lambda: moe._check(moe._lib.moe_quantize_fp8(None, 4, 16, A, A, None), "q"),       # no weights
        lambda: moe._check(moe._lib.moe_quantize_fp8(A, -1, 16, A, A, None), "q"),         # negative rows
        lambda: moe._check(moe._lib.moe_quantize_fp8(A, 4, 0, A, A, None), "q"),           # no columns
        lambda: moe.moe_expert_ffn_fp8(cfg, A, A, A, A, None, None, A, A, A, A, 0),          # SwiGLU needs W3
        lambda: moe.moe_expert_ffn_fp8(cfg, A, A, A + 8, A, A, A, A, A, A, A, 0),            # codes misaligned
        lambda: moe.moe_expert_ffn_fp8(cfg, A, A, A, None, A, A, A, A, A, A, 0),             # no scales
        lambda: moe.moe_expert_ffn_fp8(cfg, None, A, A, A, A, A, A, A, A, A, 0),             # no x_perm
        lambda: moe.moe_layer_forward_fp8(cfg, A, A, None, None, None, A, A, A, A, A, None, None, None, A, A, 0),
    ]
    for fn in invalid:
        with pytest.raises(moe.MoeError) as e:
            fn()
        assert e.value.code == moe.MOE_ERR_INVALID_ARG
    # float32 configurations and widths whose code rows are not 16-byte multiples
    for bad in (moe.make_config(64, 64, 8, 2, 128, dtype=moe.DTYPE_F32), moe.make_config(64, 72, 8, 2, 128),
                moe.make_config(64, 64, 8, 2, 136)):
        with pytest.raises(moe.MoeError) as e:
            moe.moe_expert_ffn_fp8(bad, A, A, A, A, A, A, A, A, A, A, 0)
        assert e.value.code == moe.MOE_ERR_UNSUPPORTED


def test_clock_probe_rejects_bad_arguments_without_launch():
    A = 1 << 20
    for args in ((None, 10, 1000), (A + 4, 10, 1000), (A, 1, 1000), (A, 10, 999), (A, 50002, 200_000)):
        with pytest.raises(moe.MoeError) as e:
            moe.moe_clock_probe(*args, 0)
        assert e.value.code == moe.MOE_ERR_INVALID_ARG


def test_expert_choice_config_sizes_the_workspace_for_N_times_C_rows():
    tc = moe.make_config(1000, 64, 16, 2, 128)
    ec = moe.make_config(1000, 64, 16, 1, 128, capacity=300, routing=moe.ROUTING_EXPERT_CHOICE)
    Lt, Le = moe.moe_workspace_layout(tc), moe.moe_workspace_layout(ec)
    assert Le.x_perm - Le.src_token >= 16 * 300 * 4
    assert Le.h - Le.x_perm >= 16 * 300 * 64 * 2
    assert Le.src_token - Le.dest_row >= 1000 * 16 * 4          # dest_row [T, N]
    assert Lt.src_token - Lt.dest_row >= 1000 * 2 * 4
    A = 1 << 20
    with pytest.raises(moe.MoeError):   # token-choice route on an expert-choice config
        moe.moe_route(ec, A, A, None, None, A, A, A, A, 0)
    # both dispatch entry points refuse expert choice (it dispatches in moe_ec_route)
    for fn in (lambda: moe.moe_dispatch(ec, A, A, A, A, A, A, A, A, A, 0),
               lambda: moe.moe_dispatch_noalloc(ec, A, A, A, A, A, A, A, A, None, 0)):
        with pytest.raises(moe.MoeError) as e:
            fn()
        assert e.value.code == moe.MOE_ERR_INVALID_ARG


def test_zero_tokens_is_a_noop_for_the_layer():
    cfg = moe.make_config(0, 64, 8, 2, 128)
    moe.moe_layer_forward(cfg, None, None, None, None, None, None, None, None, None, None, None, None, 0)
    moe.moe_route(cfg, None, None, None, None, None, None, None, None, 0)
    moe.moe_combine(cfg, None, None, None, None, None, 0)
