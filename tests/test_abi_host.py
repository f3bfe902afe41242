"""The C ABI on a machine without a GPU: the library loads, exports every symbol include/*.h declares, and
its host-side checks return the documented codes before anything reaches CUDA (n = 0 calls and invalid
arguments enqueue nothing)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

_abi = pytest.importorskip("decoder_attention_gb300._abi",
                           reason="libdecattn.so not built (run __graft_entry__.build())")


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\**\s*(da_\w+)\s*\(", text, flags=re.M))
    return names


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert {"da_rope_tables_build", "da_kv_cache_update", "da_attn_prefill", "da_attn_decode"} <= names
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", out, flags=re.M))
    missing = names - exported
    assert not missing, missing
    for n in names:
        getattr(_abi.LIB, n)            # resolvable through ctypes too


def test_version():
    assert _abi.version() >= 100


def _layer(**kw):
    args = dict(dtype=_abi.DA_BF16, head_dim=128, num_attention_heads=32, num_key_value_heads=8, rotary_dim=128)
    args.update(kw)
    return _abi.layer(**args)


def _rc_rope(rs, n=4):
    dummy = ctypes.c_void_p(16)
    return _abi.LIB.da_rope_tables_build(ctypes.byref(rs), dummy, dummy, n, dummy, dummy, None)


def test_rope_argument_checks():
    rs, keep = _abi.rope_scaling(1e4, 64)
    assert _rc_rope(rs, n=0) == _abi.DA_OK
    assert _rc_rope(rs, n=-1) == _abi.DA_ERR_INVALID_ARG
    rs.kind = 17
    assert _rc_rope(rs) == _abi.DA_ERR_UNSUPPORTED and "17" in _abi.last_error()
    rs, keep = _abi.rope_scaling(1e4, 63)
    assert _rc_rope(rs) == _abi.DA_ERR_INVALID_ARG
    rs, keep = _abi.rope_scaling(0.5, 64)
    assert _rc_rope(rs) == _abi.DA_ERR_INVALID_ARG
    rs, keep = _abi.rope_scaling(1e4, 64, {"type": "linear"})            # no factor
    assert _rc_rope(rs) == _abi.DA_ERR_INVALID_ARG
    rs, keep = _abi.rope_scaling(1e4, 64, {"rope_type": "llama3", "factor": 8, "low_freq_factor": 4,
                                            "high_freq_factor": 1, "original_max_position_embeddings": 8192})
    assert _rc_rope(rs) == _abi.DA_ERR_INVALID_ARG                        # high <= low
    with pytest.raises(_abi.DecAttnError):
        _abi.rope_scaling(1e4, 64, {"type": "dynamic", "factor": 2})
    sc = {"rope_type": "longrope", "short_factor": [1.0] * 32, "long_factor": [1.0] * 32,
          "original_max_position_embeddings": 4096}
    rs, keep = _abi.rope_scaling(1e4, 64, sc, 131072)
    dummy = ctypes.c_void_p(16)
    rc = _abi.LIB.da_rope_tables_build(ctypes.byref(rs), dummy, None, 4, dummy, dummy, None)
    assert rc == _abi.DA_ERR_INVALID_ARG and "seq_len" in _abi.last_error()
    bad = dict(sc, short_factor=[1.0] * 31 + [0.0])
    rs, keep = _abi.rope_scaling(1e4, 64, bad, 131072)
    assert _rc_rope(rs) == _abi.DA_ERR_INVALID_ARG


def _rc_kv(L, n=4, ptr=16):
    d = ctypes.c_void_p(ptr)
    return _abi.LIB.da_kv_cache_update(ctypes.byref(L), d, d, d, n, d, d, d, d, d, d, d, 4, 4, None)


def test_layer_argument_checks():
    assert _rc_kv(_layer(), n=0) == _abi.DA_OK
    assert _rc_kv(_layer(num_key_value_heads=5)) == _abi.DA_ERR_INVALID_ARG
    assert _rc_kv(_layer(head_dim=96, rotary_dim=96)) == _abi.DA_ERR_UNSUPPORTED
    assert _rc_kv(_layer(rotary_dim=130)) == _abi.DA_ERR_INVALID_ARG
    assert _rc_kv(_layer(rotary_dim=95)) == _abi.DA_ERR_INVALID_ARG
    assert _rc_kv(_layer(window=-1)) == _abi.DA_ERR_INVALID_ARG
    assert _rc_kv(_layer(softcap=-1.0)) == _abi.DA_ERR_INVALID_ARG
    L = _layer()
    L.q_norm_w = 64                                                        # one norm weight only
    assert _rc_kv(L) == _abi.DA_ERR_INVALID_ARG
    assert _rc_kv(_layer(), ptr=8) == _abi.DA_ERR_INVALID_ARG              # misaligned buffers
    assert _rc_kv(_layer(), n=-3) == _abi.DA_ERR_INVALID_ARG


def test_attention_argument_checks():
    L = _layer()
    d = ctypes.c_void_p(16)
    rc = _abi.LIB.da_attn_prefill(ctypes.byref(L), d, 0, d, d, 4, 4, 0, d, d, d, 0, None, d, None, 0, None)
    assert rc == _abi.DA_OK
    rc = _abi.LIB.da_attn_prefill(ctypes.byref(L), d, 8, d, d, 4, 4, -1, d, d, d, 8, None, d, None, 0, None)
    assert rc == _abi.DA_ERR_INVALID_ARG
    rc = _abi.LIB.da_attn_decode(ctypes.byref(L), d, d, d, 4, 4, 0, d, d, None, d, None, 0, None)
    assert rc == _abi.DA_OK
    rc = _abi.LIB.da_attn_decode(ctypes.byref(L), d, d, d, 0, 4, 2, d, d, None, d, None, 0, None)
    assert rc == _abi.DA_ERR_INVALID_ARG                                   # num_rows < 1
    rc = _abi.LIB.da_attn_decode(ctypes.byref(L), d, d, d, 4, 4, 2, d, None, None, d, None, 0, None)
    assert rc == _abi.DA_ERR_INVALID_ARG                                   # positions NULL


def test_decode_workspace_sizing():
    """Split plan: chunks of 512 keys grow (to 4096 at most) while the grid keeps >= 8 CTAs per SM of a
    152-SM part; workspace = S * Hq * splits * (d fp32 + (max, sum)) + 256 bytes of alignment slack."""
    L = _layer()
    ws = _abi.decode_workspace_bytes(L, 16, 131072)          # 16 x 131072 decode: 4096-key chunks, 32 splits
    assert ws == 16 * 32 * 32 * (128 * 4 + 8) + 256
    Lw = _layer(window=4096)
    ws = _abi.decode_workspace_bytes(Lw, 64, 32768)          # window 4096, 64 sequences: 1024-key chunks
    assert ws == 64 * 32 * 4 * (128 * 4 + 8) + 256
    assert _abi.decode_workspace_bytes(_layer(dtype=_abi.DA_FP32), 4, 1000) == 0   # fp32 decode needs none
    assert _abi.decode_workspace_bytes(_layer(num_key_value_heads=5), 4, 1000) == 0  # invalid layer


def test_window_for_layer():
    """DecoderConfig.window (page "42. More models", "What differs between model families")."""
    w = _abi.window_for_layer
    mistral = {"model_type": "mistral", "sliding_window": 4096, "num_hidden_layers": 4}
    assert [w(mistral, i) for i in range(4)] == [4096] * 4
    qwen2 = {"model_type": "qwen2", "sliding_window": 2048, "use_sliding_window": True, "max_window_layers": 2,
             "num_hidden_layers": 4}
    assert [w(qwen2, i) for i in range(4)] == [0, 0, 2048, 2048]
    qwen2_off = dict(qwen2, use_sliding_window=False)
    assert [w(qwen2_off, i) for i in range(4)] == [0] * 4
    gemma = {"model_type": "gemma2", "sliding_window": 4096,
             "layer_types": ["sliding_attention", "full_attention"] * 2, "num_hidden_layers": 4}
    assert [w(gemma, i) for i in range(4)] == [4096, 0, 4096, 0]
    llama = {"model_type": "llama", "sliding_window": None, "num_hidden_layers": 2}
    assert [w(llama, i) for i in range(2)] == [0, 0]


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of da_layer and da_rope_scaling have the header's size and field offsets (a C
    program built from include/decattn.h prints them)."""
    import shutil
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    structs = {"da_layer": _abi.DaLayer, "da_rope_scaling": _abi.DaRopeScaling, "da_paged_kv": _abi.DaPagedKv,
               "da_mla_layer": _abi.DaMlaLayer}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "decattn.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    cuda_inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    got = {}
    for ln in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        cname, fname, val = ln.split()
        got[(cname, fname)] = int(val)
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)


def test_mla_host_checks_and_scale():
    """MLA entry points refuse unsupported shapes before any launch; the library's softmax scale equals the
    closed form of MLAAttention (DeepSeek-V3: 192^-0.5 times (0.1 ln 40 + 1)^2)."""
    import math
    L = _abi.mla_layer(16, 0.1)
    assert _abi.LIB.da_mla_decode(ctypes.byref(L), None, None, 1, 1, 0, None, None, None, None, 0, None) == _abi.DA_OK
    bad = _abi.mla_layer(16, 0.1, kv_lora_rank=256)
    assert _abi.LIB.da_mla_decode(ctypes.byref(bad), None, None, 1, 1, 1, None, None, None, None, 0, None) == \
        _abi.DA_ERR_UNSUPPORTED
    bad = _abi.mla_layer(12, 0.1)
    assert _abi.LIB.da_mla_decode(ctypes.byref(bad), None, None, 1, 1, 1, None, None, None, None, 0, None) == \
        _abi.DA_ERR_UNSUPPORTED
    assert _abi.mla_workspace_bytes(L, 4, 1000) == 4 * 16 * 4 * (512 * 4 + 8) + 256    # 256-key chunks: 4 splits
    sc = _abi.mla_softmax_scale(128, 64, {"type": "yarn", "factor": 40, "mscale_all_dim": 1.0})
    assert abs(sc - 192 ** -0.5 * (0.1 * math.log(40) + 1) ** 2) < 1e-15
    assert math.isclose(_abi.mla_softmax_scale(128, 64), 192 ** -0.5, rel_tol=1e-15)


def test_fused_rope_update_host_checks():
    """da_kv_cache_update_rope refuses what it cannot take before anything reaches CUDA: a NULL scaling, a
    scaling whose rotary_dim differs from the layer's, layers outside bf16 / head_dim 128 / rotary_dim a
    multiple of 16, and LongRoPE without seq_len; n == 0 enqueues nothing."""
    d = ctypes.c_void_p(16)

    def rc(L, rs, n=4, seq_len=d):
        return _abi.LIB.da_kv_cache_update_rope(ctypes.byref(L), ctypes.byref(rs) if rs is not None else None, d, d, d,
                                                n, d, d, seq_len, d, d, d, 4, 4, None)
    rs, keep = _abi.rope_scaling(1e6, 128)
    assert rc(_layer(), rs, n=0) == _abi.DA_OK
    assert rc(_layer(), None) == _abi.DA_ERR_INVALID_ARG
    rs96, keep96 = _abi.rope_scaling(1e6, 96)
    assert rc(_layer(), rs96) == _abi.DA_ERR_INVALID_ARG and "rotary_dim" in _abi.last_error()
    assert rc(_layer(dtype=_abi.DA_FP32), rs) == _abi.DA_ERR_UNSUPPORTED
    rs64, keep64 = _abi.rope_scaling(1e6, 64)
    assert rc(_layer(head_dim=64, rotary_dim=64), rs64) == _abi.DA_ERR_UNSUPPORTED
    rs40, keep40 = _abi.rope_scaling(1e6, 40)
    assert rc(_layer(rotary_dim=40), rs40) == _abi.DA_ERR_UNSUPPORTED      # r/2 = 20: not a multiple of 8
    sc = {"rope_type": "longrope", "short_factor": [1.0] * 64, "long_factor": [2.0] * 64,
          "original_max_position_embeddings": 4096}
    rsl, keepl = _abi.rope_scaling(1e4, 128, sc, 131072)
    assert rc(_layer(), rsl, seq_len=None) == _abi.DA_ERR_INVALID_ARG and "seq_len" in _abi.last_error()
    assert _abi.kv_rope_fused_supported(_layer()) and not _abi.kv_rope_fused_supported(_layer(head_dim=64, rotary_dim=64))


def test_mixed_split_model():
    """da_attn_mixed_prefill_sms (host arithmetic): no hint or a decode too small to pay for the fork gives the
    prefill every SM (the parts run in turn); a decode of comparable time takes SMs from the prefill, more of
    them the more bytes it moves; the prefill keeps at least a quarter of the SMs."""
    import torch
    L = _abi.layer(torch.bfloat16, 128, 24, 8, 96, None, None, 1e-6, 0, 50.0, 0.0, None)
    pairs, keys = 8 * 1024 * 33000.0, 120 * 33000.0
    assert _abi.attn_mixed_prefill_sms(L, 152, 0.0, keys) == 152
    assert _abi.attn_mixed_prefill_sms(L, 152, pairs, 0.0) == 152
    assert _abi.attn_mixed_prefill_sms(L, 152, pairs, 8 * 4096.0) == 152
    p = [_abi.attn_mixed_prefill_sms(L, 152, pairs, keys * f) for f in (0.5, 1.0, 1.5)]
    assert all(152 // 4 <= x < 152 for x in p), p
    assert p[0] >= p[1] >= p[2], p
    assert 76 // 4 <= _abi.attn_mixed_prefill_sms(L, 76, pairs, keys) <= 76
    for bad in ((152, float("nan"), keys), (152, -1.0, keys), (0, pairs, keys)):
        with pytest.raises(_abi.DecAttnError):
            _abi.attn_mixed_prefill_sms(L, *bad)


def test_mixed_argument_checks():
    L = _layer()
    d = ctypes.c_void_p(16)
    P = ctypes.c_double
    rc = _abi.LIB.da_attn_mixed(ctypes.byref(L), d, d, d, 4, 4, 8, 1, d, d, d, 8, -1, d, d, P(0), P(0), d, None, 0,
                                None)
    assert rc == _abi.DA_ERR_INVALID_ARG                                   # n_decode < 0
    rc = _abi.LIB.da_attn_mixed(ctypes.byref(L), d, d, d, 4, 4, 8, 1, d, d, d, 8, 2, d, d, P(float("nan")), P(0), d,
                                None, 0, None)
    assert rc == _abi.DA_ERR_INVALID_ARG                                   # hint not finite
    rc = _abi.LIB.da_attn_mixed(None, d, d, d, 4, 4, 8, 1, d, d, d, 8, 2, d, d, P(0), P(0), d, None, 0, None)
    assert rc == _abi.DA_ERR_INVALID_ARG                                   # no layer
