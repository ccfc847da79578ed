"""The C-ABI library loads, exports every entry point include/moe.h declares,
and its host-side validation rejects bad arguments (no GPU needed)."""
import ctypes
import os
import re

import pytest

import quantized_expert_ffn_softmax_gb300 as moe
from quantized_expert_ffn_softmax_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "moe_forward" in names and "moe_layer_create" in names
    raw = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_version_and_empty_error(lib):
    assert moe.moe_version() == 300
    assert isinstance(moe.moe_last_error(), str)


def _cfg(**kw):
    c = dict(hidden=256, n_experts=16, top_k=2, ffn=128, shared_ffn=128, max_tokens=8)
    c.update(kw)
    return c


@pytest.mark.parametrize("bad", [dict(hidden=100), dict(hidden=0), dict(n_experts=0),
                                 dict(n_experts=2000), dict(top_k=0), dict(top_k=17),
                                 dict(top_k=20, n_experts=16), dict(ffn=96), dict(shared_ffn=64),
                                 dict(max_tokens=0), dict(n_slots=7), dict(n_slots=17), dict(routing_flags=8),
                                 dict(routing_flags=-1), dict(routing_flags=4, shared_ffn=0)])
def test_create_rejects_bad_configs_before_touching_the_device(lib, bad):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_create(_cfg(**bad), {}, False)
    assert ei.value.status == moe.MOE_ERR_INVALID


def test_create_rejects_missing_weights(lib):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_create(_cfg(), {"router_w": 1}, False)
    assert ei.value.status == moe.MOE_ERR_INVALID
    assert "NULL" in moe.moe_last_error()


def test_calls_reject_null_layer(lib):
    L = lib
    assert L.moe_forward(None, None, 1, None, None) == moe.MOE_ERR_INVALID
    assert L.moe_route(None, None, 1, None, None, None) == moe.MOE_ERR_INVALID
    assert L.moe_status_sync(None, None) == moe.MOE_ERR_INVALID
    arr = (ctypes.c_void_p * 1)(None)
    assert L.moe_stack_forward(arr, 0, None, 1, None, None) == moe.MOE_ERR_INVALID
    L.moe_layer_destroy(None)


def test_create_refuses_shapes_whose_single_token_decode_cannot_fit(lib):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_create(_cfg(hidden=8192, n_experts=256, top_k=8, ffn=512, shared_ffn=512), {}, False)
    assert ei.value.status == moe.MOE_ERR_INVALID
    assert "shared memory" in moe.moe_last_error()
    # the benchmarked shapes pass the shape checks (and stop at the missing weights)
    for shape in (dict(hidden=2048, n_experts=256, top_k=8, ffn=512, shared_ffn=512),
                  dict(hidden=2048, n_experts=512, top_k=10, ffn=768, shared_ffn=1536),
                  dict(hidden=2048, n_experts=512, top_k=10, ffn=768, shared_ffn=1536,
                       routing_flags=7)):
        with pytest.raises(moe.MoeError):
            moe.moe_layer_create(_cfg(**shape), {}, False)
        assert "NULL" in moe.moe_last_error()


def test_create_requires_the_gate_vector_of_a_gated_shared_expert(lib):
    names = ("router_w", "router_bias", "slot_of_expert", "gate_q", "gate_s", "up_q", "up_s",
             "down_q", "down_s", "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q",
             "sh_down_s")
    fake = {n: 16 for n in names}  # non-null placeholders: refused before any device access
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_create(_cfg(routing_flags=moe.ROUTING_SHARED_GATE), fake, False)
    assert ei.value.status == moe.MOE_ERR_INVALID
    assert "sh_gate_w" in moe.moe_last_error()
