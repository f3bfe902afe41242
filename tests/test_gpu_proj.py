"""The projections around the step on the GPU against the oracle: the fused q/k/v projection (GEMM with the
norm, RoPE and cache write in its epilogue) and o_proj (plain GEMM), at small sizes whole (ragged token tiles,
biases, norm weights, paged pools) and at the Qwen3-8B shape on sampled tokens."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import proj as P

pytestmark = pytest.mark.gpu


def _rope_tables(positions, d, theta):
    inv, af = A.rope_inv_freq(d, theta, None, None)
    return A.rope_tables(np.asarray(positions), inv, af)


def _setup(n, hidden, hq, hkv, R, M, seed, norm=True, bias=True):
    g = torch.Generator().manual_seed(seed)
    d = 128
    x = torch.randn((n, hidden), generator=g).to(torch.bfloat16)
    w = (torch.randn(((hq + 2 * hkv) * d, hidden), generator=g) / math.sqrt(hidden)).to(torch.bfloat16)
    b = torch.randn((hq + 2 * hkv) * d, generator=g) * 0.1 if bias else None
    qn = (1 + 0.1 * torch.randn(d, generator=g)) if norm else None
    kn = (1 + 0.1 * torch.randn(d, generator=g)) if norm else None
    slots = torch.randperm(R * M, generator=g)[:n]
    rows, pos = (slots // M).to(torch.int32), (slots % M).to(torch.int32)
    kc = torch.randn((R, hkv, M, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((R, hkv, M, d), generator=g).to(torch.bfloat16)
    return x, w, b, qn, kn, rows, pos, kc, vc


def _layer(hq, hkv, qn, kn, cuda):
    from decoder_attention_gb300 import _abi
    qd = qn.to(cuda).float().contiguous() if qn is not None else None
    kd = kn.to(cuda).float().contiguous() if kn is not None else None
    return _abi.layer(torch.bfloat16, 128, hq, hkv, 128, qd, kd, 1e-6), (qd, kd)


@pytest.mark.parametrize("n,norm,bias", [(300, True, True), (128, False, False), (1, True, False)])
def test_fused_qkv_matches_oracle(cuda, n, norm, bias):
    from decoder_attention_gb300 import _abi
    hidden, hq, hkv, R, M = 256, 4, 2, 3, 200
    x, w, b, qn, kn, rows, pos, kc, vc = _setup(n, hidden, hq, hkv, R, M, seed=n, norm=norm, bias=bias)
    cos, sin = _rope_tables(pos.numpy(), 128, 1e6)
    layer = A.Layer(head_dim=128, num_attention_heads=hq, num_key_value_heads=hkv, rotary_dim=128,
                    q_norm_w=qn.double().numpy() if norm else None, k_norm_w=kn.double().numpy() if norm else None)
    kc64, vc64 = kc.double().numpy().copy(), vc.double().numpy().copy()
    q_ref = P.project_and_update(layer, x.double().numpy(), w.double().numpy(), rows.numpy(), pos.numpy(), cos, sin,
                                 kc64, vc64, b.double().numpy() if bias else None)
    L, keep = _layer(hq, hkv, qn, kn, cuda)
    xd, wd = x.to(cuda), w.to(cuda)
    bd = b.to(cuda).float() if bias else None
    kcd, vcd = kc.to(cuda), vc.to(cuda)
    q_rot = torch.empty((n, hq, 128), dtype=torch.bfloat16, device=cuda)
    cd = torch.from_numpy(cos).float().to(cuda)
    sd = torch.from_numpy(sin).float().to(cuda)
    _abi.qkv_project_update(L, xd, wd, bd, n, hidden, rows.to(cuda), pos.to(cuda), cd, sd, q_rot, kcd, vcd, R, M)
    torch.cuda.synchronize()
    _abi.check_device_error()
    np.testing.assert_allclose(q_rot.double().cpu().numpy(), q_ref, rtol=2.0 ** -7, atol=2e-3)
    written = torch.zeros((R, M), dtype=torch.bool)
    written[rows.long(), pos.long()] = True
    kg, vg = kcd.cpu(), vcd.cpu()
    r_i, p_i = rows.numpy().astype(np.int64), pos.numpy().astype(np.int64)
    np.testing.assert_allclose(kg.double().numpy()[r_i, :, p_i], kc64[r_i, :, p_i], rtol=2.0 ** -7, atol=2e-3)
    np.testing.assert_allclose(vg.double().numpy()[r_i, :, p_i], vc64[r_i, :, p_i], rtol=2.0 ** -7, atol=2e-3)
    w4 = written[:, None, :, None].expand_as(kg)
    assert torch.equal(kg[~w4], kc[~w4]) and torch.equal(vg[~w4], vc[~w4])


def test_fused_qkv_paged(cuda):
    from decoder_attention_gb300 import _abi, inputs
    hidden, hq, hkv, R, M, n = 256, 4, 2, 3, 256, 200
    x, w, b, qn, kn, rows, pos, kc, vc = _setup(n, hidden, hq, hkv, R, M, seed=7)
    cos, sin = _rope_tables(pos.numpy(), 128, 1e6)
    layer = A.Layer(head_dim=128, num_attention_heads=hq, num_key_value_heads=hkv, rotary_dim=128,
                    q_norm_w=qn.double().numpy(), k_norm_w=kn.double().numpy())
    kc64, vc64 = kc.double().numpy().copy(), vc.double().numpy().copy()
    q_ref = P.project_and_update(layer, x.double().numpy(), w.double().numpy(), rows.numpy(), pos.numpy(), cos, sin,
                                 kc64, vc64, b.double().numpy())
    kp, vp, table = inputs.paged_from_contiguous(kc.to(cuda), vc.to(cuda), 64, seed=3, spare_blocks=2)
    kv = _abi.paged_kv(kp, vp, table, 64)
    L, keep = _layer(hq, hkv, qn, kn, cuda)
    q_rot = torch.empty((n, hq, 128), dtype=torch.bfloat16, device=cuda)
    _abi.qkv_project_update_paged(L, x.to(cuda), w.to(cuda), b.to(cuda).float(), n, hidden, rows.to(cuda),
                                  pos.to(cuda), torch.from_numpy(cos).float().to(cuda),
                                  torch.from_numpy(sin).float().to(cuda), q_rot, kv)
    torch.cuda.synchronize()
    _abi.check_device_error()
    np.testing.assert_allclose(q_rot.double().cpu().numpy(), q_ref, rtol=2.0 ** -7, atol=2e-3)
    t = table.cpu().numpy()
    kpc = kp.double().cpu().numpy()
    for i in range(n):
        r, p = int(rows[i]), int(pos[i])
        np.testing.assert_allclose(kpc[t[r, p // 64], :, p % 64], kc64[r, :, p], rtol=2.0 ** -7, atol=2e-3)


@pytest.mark.parametrize("m,n,k,bias", [(300, 512, 1024, True), (128, 256, 64, False)])
def test_linear_matches_oracle(cuda, m, n, k, bias):
    from decoder_attention_gb300 import _abi
    g = torch.Generator().manual_seed(m + n)
    x = torch.randn((m, k), generator=g).to(torch.bfloat16)
    w = (torch.randn((n, k), generator=g) / math.sqrt(k)).to(torch.bfloat16)
    b = torch.randn(n, generator=g) if bias else None
    y = torch.empty((m, n), dtype=torch.bfloat16, device=cuda)
    _abi.linear(x.to(cuda), w.to(cuda), b.to(cuda).float() if bias else None, m, n, k, y)
    torch.cuda.synchronize()
    ref = P.o_project(x.double().numpy().reshape(m, 1, k), w.double().numpy(), b.double().numpy() if bias else None)
    np.testing.assert_allclose(y.double().cpu().numpy(), ref, rtol=2.0 ** -7, atol=2e-3)


def test_qwen3_shape_sampled(cuda):
    """Qwen3-8B shapes (8192 tokens, hidden 4096, Hq 32, Hkv 8, q/k norm): fused projection and o_proj, 48
    sampled tokens checked against the oracle."""
    from decoder_attention_gb300 import _abi
    n, hidden, hq, hkv, R, M = 8192, 4096, 32, 8, 4, 2048
    g = torch.Generator(device=cuda).manual_seed(11)
    x = torch.randn((n, hidden), generator=g, device=cuda).to(torch.bfloat16)
    w = (torch.randn(((hq + 2 * hkv) * 128, hidden), generator=g, device=cuda) / 64).to(torch.bfloat16)
    qn = 1 + 0.1 * torch.randn(128, generator=g, device=cuda)
    kn = 1 + 0.1 * torch.randn(128, generator=g, device=cuda)
    rows = (torch.arange(n, device=cuda) // M).to(torch.int32)
    pos = (torch.arange(n, device=cuda) % M).to(torch.int32)
    kc = torch.zeros((R, hkv, M, 128), dtype=torch.bfloat16, device=cuda)
    vc = torch.zeros_like(kc)
    cos, sin = _rope_tables(pos.cpu().numpy(), 128, 1e6)
    cd, sd = torch.from_numpy(cos).float().to(cuda), torch.from_numpy(sin).float().to(cuda)
    L = _abi.layer(torch.bfloat16, 128, hq, hkv, 128, qn, kn, 1e-6)
    q_rot = torch.empty((n, hq, 128), dtype=torch.bfloat16, device=cuda)
    _abi.qkv_project_update(L, x, w, None, n, hidden, rows, pos, cd, sd, q_rot, kc, vc, R, M)
    wo = (torch.randn((hidden, hq * 128), generator=g, device=cuda) / 64).to(torch.bfloat16)
    y = torch.empty((n, hidden), dtype=torch.bfloat16, device=cuda)
    _abi.linear(q_rot.view(n, hq * 128), wo, None, n, hidden, hq * 128, y)
    torch.cuda.synchronize()
    _abi.check_device_error()
    layer = A.Layer(head_dim=128, num_attention_heads=hq, num_key_value_heads=hkv, rotary_dim=128,
                    q_norm_w=qn.double().cpu().numpy(), k_norm_w=kn.double().cpu().numpy())
    idx = torch.randperm(n, generator=torch.Generator().manual_seed(2))[:48].sort().values.numpy()
    xs = x.double().cpu().numpy()[idx]
    kc64, vc64 = np.zeros((R, hkv, M, 128)), np.zeros((R, hkv, M, 128))
    q_ref = P.project_and_update(layer, xs, w.double().cpu().numpy(), rows.cpu().numpy()[idx], pos.cpu().numpy()[idx],
                                 cos[idx], sin[idx], kc64, vc64)
    np.testing.assert_allclose(q_rot.double().cpu().numpy()[idx], q_ref, rtol=2.0 ** -7, atol=4e-3)
    r_i, p_i = rows.cpu().numpy()[idx], pos.cpu().numpy()[idx]
    np.testing.assert_allclose(kc.double().cpu().numpy()[r_i, :, p_i], kc64[r_i, :, p_i], rtol=2.0 ** -7, atol=4e-3)
    np.testing.assert_allclose(vc.double().cpu().numpy()[r_i, :, p_i], vc64[r_i, :, p_i], rtol=2.0 ** -7, atol=4e-3)
    y_ref = P.o_project(q_rot.double().cpu().numpy()[idx], wo.double().cpu().numpy())
    np.testing.assert_allclose(y.double().cpu().numpy()[idx], y_ref, rtol=2.0 ** -7, atol=4e-3)


def test_fused_qkv_invalid_token(cuda):
    """A token whose position is past the cache: the device error word says so and no cache slot is written for
    it; its q_rot and every other token's outputs are still correct."""
    from decoder_attention_gb300 import _abi
    hidden, hq, hkv, R, M, n = 256, 4, 2, 3, 200, 150
    x, w, b, qn, kn, rows, pos, kc, vc = _setup(n, hidden, hq, hkv, R, M, seed=11)
    bad_pos = pos.clone()
    bad_pos[37] = M                                   # one past the last slot
    cos, sin = _rope_tables(pos.numpy(), 128, 1e6)    # the rotation itself is the valid position's
    layer = A.Layer(head_dim=128, num_attention_heads=hq, num_key_value_heads=hkv, rotary_dim=128,
                    q_norm_w=qn.double().numpy(), k_norm_w=kn.double().numpy())
    kc64, vc64 = kc.double().numpy().copy(), vc.double().numpy().copy()
    q_ref = P.project_and_update(layer, x.double().numpy(), w.double().numpy(), rows.numpy(), pos.numpy(), cos, sin,
                                 kc64, vc64, b.double().numpy())
    L, keep = _layer(hq, hkv, qn, kn, cuda)
    kcd, vcd = kc.to(cuda), vc.to(cuda)
    q_rot = torch.empty((n, hq, 128), dtype=torch.bfloat16, device=cuda)
    _abi.qkv_project_update(L, x.to(cuda), w.to(cuda), b.to(cuda).float(), n, hidden, rows.to(cuda),
                            bad_pos.to(cuda), torch.from_numpy(cos).float().to(cuda),
                            torch.from_numpy(sin).float().to(cuda), q_rot, kcd, vcd, R, M)
    torch.cuda.synchronize()
    with pytest.raises(_abi.DecAttnError) as ei:
        _abi.check_device_error()
    assert ei.value.code == _abi.DA_ERR_DEVICE_INDEX
    np.testing.assert_allclose(q_rot.double().cpu().numpy(), q_ref, rtol=2.0 ** -7, atol=2e-3)
    ok = np.arange(n) != 37
    r_i, p_i = rows.numpy().astype(np.int64)[ok], pos.numpy().astype(np.int64)[ok]
    kg, vg = kcd.cpu(), vcd.cpu()
    np.testing.assert_allclose(kg.double().numpy()[r_i, :, p_i], kc64[r_i, :, p_i], rtol=2.0 ** -7, atol=2e-3)
    np.testing.assert_allclose(vg.double().numpy()[r_i, :, p_i], vc64[r_i, :, p_i], rtol=2.0 ** -7, atol=2e-3)
    r37, p37 = int(rows[37]), int(pos[37])           # the slot the token would have had is untouched
    assert torch.equal(kg[r37, :, p37], kc[r37, :, p37]) and torch.equal(vg[r37, :, p37], vc[r37, :, p37])
    _abi.check_device_error()
