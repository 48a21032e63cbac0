"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element.

Small cases compare every element of O, L, dQ, dK and dV with the full oracle.
At the full workload sizes the oracle checks whole sampled heads plus sampled
query rows (O, L, dQ) and key rows (dK, dV); the causal N=65536 case checks
sampled rows and, over every key, the sum rules that hold at any size.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_97_gb300.inputs import WORKLOADS, make_qkv_do, sample_indices

from parity import check, run_gpu

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.float().double().numpy()


def _full_ref(q, k, v, dO, scale, causal):
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, scale, causal)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def _as_dict(res):
    return dict(zip(("o", "lse", "dq", "dk", "dv"), res))


# ------------------------------------------------------------ worked examples (fp32 path)

def test_tutorial_row_on_gpu():
    g = json.load(open(os.path.join(GOLDEN, "tutorial_single_row.json")))
    s = torch.tensor(g["scores"], dtype=torch.float32)
    q = torch.tensor([[1.0, 0.0]] * 4).view(1, 1, 4, 2)
    k = torch.stack([s, torch.zeros(4)], dim=1).view(1, 1, 4, 2)
    v = torch.tensor(g["values"]).view(1, 1, 4, 2)
    dO = torch.ones_like(v)
    got = _as_dict(run_gpu(q, k, v, dO, 1.0, False))
    check("tutorial_row_f32", "f32", got, _full_ref(_np(q), _np(k), _np(v), _np(dO), 1.0, False))
    for i in range(4):
        assert np.max(np.abs(got["o"][0, 0, i] - g["printed_output"])) <= 5e-7 + 1e-6


def test_llama_notes_example_on_gpu():
    g = json.load(open(os.path.join(GOLDEN, "llama_notes_four_tokens.json")))
    X = torch.tensor(g["X"], dtype=torch.float32).view(1, 1, 4, 2)
    scale = 1.0 / math.sqrt(2.0)
    dO = torch.tensor([[1.0, -1.0], [0.5, 2.0], [-1.0, 0.0], [0.25, 0.25]]).view(1, 1, 4, 2)
    for causal in (False, True):
        got = _as_dict(run_gpu(X, X, X, dO, scale, causal))
        check(f"llama_notes_f32_causal{int(causal)}", "f32", got,
              _full_ref(_np(X), _np(X), _np(X), _np(dO), scale, causal))
    got = _as_dict(run_gpu(X, X, X, dO, scale, False))
    assert np.max(np.abs(got["o"][0, 0, 0] - g["output_token0"])) <= g["tol_outputs"]
    assert np.max(np.abs(got["o"][0, 0, 1] - g["output_token1"])) <= g["tol_outputs"]
    assert abs(math.exp(got["lse"][0, 0, 0]) - g["denominator_row0"]) <= g["tol_sums"]


# ------------------------------------------------------------ fp32 path

def test_f32_B1_H2_N256_d64():
    w = WORKLOADS["f32_B1_H2_N256_d64"]
    q, k, v, dO = make_qkv_do(w.B, w.H, w.N, w.d, w.seed, torch.float32)
    got = _as_dict(run_gpu(q, k, v, dO, w.scale, w.causal))
    check(w.name, "f32", got, _full_ref(_np(q), _np(k), _np(v), _np(dO), w.scale, w.causal))


@pytest.mark.parametrize("d", [1, 3, 17, 64, 100, 128])
@pytest.mark.parametrize("N", [1, 5, 33, 130])
@pytest.mark.parametrize("causal", [False, True])
def test_f32_ragged(d, N, causal):
    q, k, v, dO = make_qkv_do(2, 1, N, d, seed=7 * d + N, dtype=torch.float32)
    got = _as_dict(run_gpu(q, k, v, dO, 1.0 / math.sqrt(d), causal))
    check(f"f32_ragged_N{N}_d{d}_c{int(causal)}", "f32", got,
          _full_ref(_np(q), _np(k), _np(v), _np(dO), 1.0 / math.sqrt(d), causal))


# ------------------------------------------------------------ bf16 tensor-core path, full oracle

@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("N", [1, 4, 127, 128, 129, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_small_and_ragged(d, N, causal):
    q, k, v, dO = make_qkv_do(1, 2, N, d, seed=1000 + N + d, dtype=torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    got = _as_dict(run_gpu(q, k, v, dO, scale, causal))
    check(f"bf16_small_N{N}_d{d}_c{int(causal)}", "bf16", got,
          _full_ref(_np(q), _np(k), _np(v), _np(dO), scale, causal))


@pytest.mark.parametrize("d", [64, 96, 128])
def test_bf16_scale_and_large_scores(d):
    """Scores far from the unit range (the running max moves by many 2^8
    steps): a large scale and queries scaled up."""
    q, k, v, dO = make_qkv_do(1, 2, 700, d, seed=55, dtype=torch.float32)
    q = (q * 4).to(torch.bfloat16)
    k, v, dO = (x.to(torch.bfloat16) for x in (k, v, dO))
    for causal in (False, True):
        got = _as_dict(run_gpu(q, k, v, dO, 0.5, causal))
        check(f"bf16_large_scores_d{d}_c{int(causal)}", "bf16", got,
              _full_ref(_np(q), _np(k), _np(v), _np(dO), 0.5, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_B2_H4_N1000_d96(causal):
    """Head size 96: tiles are padded to two 64-column boxes, products use
    N = 96; many tiles per item and a ragged tail."""
    q, k, v, dO = make_qkv_do(2, 4, 1000, 96, seed=96, dtype=torch.bfloat16)
    scale = 1.0 / math.sqrt(96)
    got = _as_dict(run_gpu(q, k, v, dO, scale, causal))
    check(f"bf16_B2_H4_N1000_d96_c{int(causal)}", "bf16", got,
          _full_ref(_np(q), _np(k), _np(v), _np(dO), scale, causal))


@pytest.mark.parametrize("N,causal", [(1, False), (300, False), (300, True), (700, True)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_fwd_d256(N, causal, dtype):
    """Head size 256, forward only: K and V stream as two 128-column units
    per key tile; the backward refuses d = 256."""
    import exact_attention_97_gb300 as fa
    q, k, v, dO = make_qkv_do(1, 3, N, 256, seed=256 + N, dtype=dtype)
    scale = 1.0 / math.sqrt(256)
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o, lse = fa.attention_forward(qd, kd, vd, scale, causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ro, rl = oracle.attention_fwd(_np(q), _np(k), _np(v), scale, causal)
    check(f"fwd_d256_N{N}_c{int(causal)}_{str(dtype)[6:]}", "bf16",
          {"o": o.float().cpu().double().numpy(), "lse": lse.cpu().double().numpy()}, {"o": ro, "lse": rl})
    with pytest.raises(fa.FAError):
        fa.attention_backward(qd, kd, vd, o, lse, dO.to(dev), scale, causal)


def test_fwd_d256_kv():
    import exact_attention_97_gb300 as fa
    q, _, _, _ = make_qkv_do(2, 2, 130, 256, seed=7, dtype=torch.bfloat16)
    _, k, v, _ = make_qkv_do(2, 2, 900, 256, seed=8, dtype=torch.bfloat16)
    scale = 1.0 / math.sqrt(256)
    dev = torch.device("cuda")
    o, lse = fa.attention_forward(q.to(dev), k.to(dev), v.to(dev), scale, True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ro, rl = oracle.attention_fwd_kv(_np(q), _np(k), _np(v), scale, True)
    check("fwd_d256_kv_Nq130_Nk900_c1", "bf16",
          {"o": o.float().cpu().double().numpy(), "lse": lse.cpu().double().numpy()}, {"o": ro, "lse": rl})


# ------------------------------------------------------------ persistent schedule, several items per CTA

@pytest.mark.parametrize("B,H,Nq,Nk,d", [
    (2, 24, 2048, 2048, 64),   # pairs of query tiles / key blocks, then single tiles of the last 19 heads
    (2, 20, 1000, 4000, 64),   # snake order over unequal causal costs (bottom-right mask)
    (2, 30, 1400, 1400, 64),   # 11 tiles per head: pair units with an odd middle tile (empty slots)
])
def test_causal_schedules_with_several_items_per_cta(B, H, Nq, Nk, d):
    """The host picks the schedule mode from exact tile costs (the CPU test
    checks which one for these shapes); every item of every CTA must land
    once, whatever the mode."""
    q, _, _, dO = make_qkv_do(B, H, Nq, d, seed=600 + Nq, dtype=torch.bfloat16)
    _, k, v, _ = make_qkv_do(B, H, Nk, d, seed=700 + Nk, dtype=torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    got = _run_gpu_kv(q, k, v, dO, scale, True)
    o, lse = oracle.attention_fwd_kv(_np(q), _np(k), _np(v), scale, True)
    dq, dk, dv = oracle.attention_bwd_kv(_np(q), _np(k), _np(v), _np(dO), scale, True)
    check(f"sched_B{B}_H{H}_Nq{Nq}_Nk{Nk}_d{d}", "bf16", got, {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv})


@pytest.mark.parametrize("B,H,Nq,Nk,causal", [
    (2, 24, 2048, 2048, True),   # 8 tile pairs / key-block pairs per head, several per cluster
    (2, 12, 1100, 1300, True),   # 9 query tiles and 11 key blocks: each head's last pair has one tile
    (3, 5, 1100, 1300, False),   # the same without the mask
])
def test_d128_several_items_per_cta(B, H, Nq, Nk, causal):
    """Head size 128 with several items per persistent CTA and odd tile and
    block counts (the two-CTA variant of these kernels runs the same shapes
    in test_gpu_pair_kernels.py)."""
    q, _, _, dO = make_qkv_do(B, H, Nq, 128, seed=800 + Nq + B, dtype=torch.bfloat16)
    _, k, v, _ = make_qkv_do(B, H, Nk, 128, seed=900 + Nk + B, dtype=torch.bfloat16)
    scale = 1.0 / math.sqrt(128)
    got = _run_gpu_kv(q, k, v, dO, scale, causal)
    o, lse = oracle.attention_fwd_kv(_np(q), _np(k), _np(v), scale, causal)
    dq, dk, dv = oracle.attention_bwd_kv(_np(q), _np(k), _np(v), _np(dO), scale, causal)
    check(f"pair_B{B}_H{H}_Nq{Nq}_Nk{Nk}_c{int(causal)}", "bf16", got,
          {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv})


# ------------------------------------------------------------ host-resident training step

@pytest.mark.parametrize("case", ["bf16_causal", "f16_kv", "dropout", "one_chunk", "sizes"])
def test_host_step_equals_device_path(case):
    """attention_step_host streams chunks of heads through the GPU on three
    streams; its results must equal the device-side calls bit for bit."""
    import exact_attention_97_gb300 as fa
    dt = torch.float16 if case == "f16_kv" else torch.bfloat16
    Nk = 700 if case == "f16_kv" else 300
    q, _, _, dO = make_qkv_do(2, 5, 300, 128, seed=77, dtype=dt)
    _, k, v, _ = make_qkv_do(2, 5, Nk, 128, seed=78, dtype=dt)
    kw = {"dropout_p": 0.2, "seed": 5, "offset": 1} if case == "dropout" else {}
    chunks = {"one_chunk": 1, "sizes": [1, 3, 4, 2]}.get(case, 4)
    pin = [t.pin_memory() for t in (q, k, v, dO)]
    res = fa.attention_step_host(*pin, None, True, chunks=chunks, **kw)
    torch.cuda.current_stream().synchronize()
    dev = [t.cuda() for t in (q, k, v, dO)]
    o, lse = fa.attention_forward(*dev[:3], None, True, **kw)
    g = fa.attention_backward(*dev[:3], o, lse, dev[3], None, True, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for a, b in zip(res, (o, lse, *g)):
        assert torch.equal(a, b.cpu())


@pytest.mark.parametrize("case", ["bf16_causal", "f16_kv", "dropout_saved", "f32"])
def test_autograd_attention_equals_the_direct_calls(case):
    """fa.attention through torch.autograd: O and the gradients that
    .backward() produces equal attention_forward / attention_backward on the
    same dO, bit for bit (same kernels, same arguments). The fp32 backward
    sums dK and dV with atomic adds, whose order varies from run to run, so
    its gradients are compared to 1e-5 of their largest magnitude."""
    import exact_attention_97_gb300 as fa
    dt = {"f16_kv": torch.float16, "f32": torch.float32}.get(case, torch.bfloat16)
    Nk = 700 if case == "f16_kv" else 300
    d = 64 if case == "f32" else 128
    q, _, _, dO = make_qkv_do(2, 3, 300, d, seed=91, dtype=dt)
    _, k, v, _ = make_qkv_do(2, 3, Nk, d, seed=92, dtype=dt)
    q, k, v, dO = (t.cuda() for t in (q, k, v, dO))
    kw = dict(dropout_p=0.2, seed=9, offset=1) if case == "dropout_saved" else {}
    qa, ka, va = (t.clone().requires_grad_() for t in (q, k, v))
    o, lse = fa.attention(qa, ka, va, None, True, save_dropout_mask=case == "dropout_saved", return_lse=True, **kw)
    assert not lse.requires_grad
    o.backward(dO)
    o2, lse2 = fa.attention_forward(q, k, v, None, True, **kw)
    g2 = fa.attention_backward(q, k, v, o2, lse2, dO, None, True, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    assert torch.equal(o.detach(), o2) and torch.equal(lse, lse2)
    for a, b in zip((qa.grad, ka.grad, va.grad), g2):
        if case == "f32":
            assert float((a - b).abs().max()) <= 1e-5 * float(b.abs().max())
        else:
            assert torch.equal(a, b)


# ------------------------------------------------------------ dropout

def _drop_ref(q, k, v, dO, scale, causal, seed, offset, p):
    t = oracle.dropout_threshold(p)
    o, lse = oracle.attention_fwd_dropout_kv(_np(q), _np(k), _np(v), scale, causal, seed, offset, t)
    ref = {"o": o, "lse": lse}
    if dO is not None:
        dq, dk, dv = oracle.attention_bwd_dropout_kv(_np(q), _np(k), _np(v), _np(dO), scale, causal, seed, offset, t)
        ref.update(dq=dq, dk=dk, dv=dv)
    return ref


def _run_drop(q, k, v, dO, scale, causal, seed, offset, p, plain_workspace=False):
    """Forward (and backward) with drawn keep bits. By default the backward's
    workspace has room for the bits, so its dQ pass reads those its dK/dV
    pass drew; plain_workspace=True makes the dQ pass draw them itself."""
    import exact_attention_97_gb300 as fa
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    o, lse = fa.attention_forward(qd, kd, vd, scale, causal, dropout_p=p, seed=seed, offset=offset)
    got = {"o": o, "lse": lse}
    if dO is not None:
        ws = None
        if plain_workspace:
            B, H, Nq, d = q.shape
            kind = fa.FA_F16 if q.dtype == torch.float16 else fa.FA_BF16
            ws = torch.empty(fa.fa_bwd_workspace_size(B, H, Nq, d, kind), device=dev, dtype=torch.uint8)
        dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dO.to(dev), scale, causal, dropout_p=p, seed=seed,
                                           offset=offset, workspace=ws)
        got.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return {key: t.float().cpu().double().numpy() for key, t in got.items()}


def _mask(seed, offset, p, B, H, Nq, Nk, causal):
    t = oracle.dropout_threshold(p)
    m = np.stack([oracle.dropout_mask(seed, offset, t, h, Nq, Nk) for h in range(B * H)]).reshape(B, H, Nq, Nk)
    if causal:
        i = np.arange(Nq)[:, None]
        j = np.arange(Nk)[None, :]
        m = m * (j <= i + (Nk - Nq))
    return m.astype(bool)


@pytest.mark.parametrize("d,Nq,Nk,causal", [(128, 300, 128, False), (128, 100, 128, True), (256, 200, 256, False),
                                            (256, 130, 256, True)])
def test_dropout_forward_mask_is_exact(d, Nq, Nk, causal):
    """With V the identity (value j = unit vector j, Nk <= d), O[i, j] is the
    kept-and-scaled probability P[i, j] Z[i, j] / (1 - p): its zero pattern is
    the mask, which must equal the oracle's bit for bit."""
    seed, offset, p = 0x5EED5EED1234, 3, 0.3
    q, k, _, _ = make_qkv_do(1, 3, Nq, d, seed=7, dtype=torch.float32)
    _, k, _, _ = make_qkv_do(1, 3, Nk, d, seed=8, dtype=torch.float32)
    q, k = (0.2 * q).to(torch.bfloat16), (0.2 * k).to(torch.bfloat16)  # scores near 0: no P underflows
    v = torch.zeros(1, 3, Nk, d)
    v[:, :, torch.arange(Nk), torch.arange(Nk)] = 1.0
    v = v.to(torch.bfloat16)
    got = _run_drop(q, k, v, None, 1.0 / math.sqrt(d), causal, seed, offset, p)
    want = _mask(seed, offset, p, 1, 3, Nq, Nk, causal)
    assert np.array_equal(got["o"][..., :Nk] != 0, want)
    check(f"dropout_fwd_identity_d{d}_Nq{Nq}_c{int(causal)}", "bf16", got,
          _drop_ref(q, k, v, None, 1.0 / math.sqrt(d), causal, seed, offset, p))


@pytest.mark.parametrize("Nk", [128, 300, 513])
def test_dropout_dkdv_mask_is_exact(Nk):
    """dV = (P o Z / (1 - p))^T dO with dO the identity (Nq = d = 128): the
    zero pattern of dV^T is the mask, drawn in the dK/dV pass's key-owner
    layout, across several key blocks."""
    seed, offset, p = 77, 11, 0.25
    q, _, _, _ = make_qkv_do(1, 2, 128, 128, seed=9, dtype=torch.float32)
    _, k, v, _ = make_qkv_do(1, 2, Nk, 128, seed=10, dtype=torch.float32)
    q, k, v = (0.2 * q).to(torch.bfloat16), (0.2 * k).to(torch.bfloat16), v.to(torch.bfloat16)
    dO = torch.eye(128).expand(1, 2, 128, 128).contiguous().to(torch.bfloat16)
    got = _run_drop(q, k, v, dO, 1.0 / math.sqrt(128), False, seed, offset, p)
    want = _mask(seed, offset, p, 1, 2, 128, Nk, False)
    assert np.array_equal(np.swapaxes(got["dv"], 2, 3)[..., :128, :] != 0, want)
    check(f"dropout_dkdv_identity_Nk{Nk}", "bf16", got,
          _drop_ref(q, k, v, dO, 1.0 / math.sqrt(128), False, seed, offset, p))


@pytest.mark.parametrize("plain_workspace", [False, True])
def test_dropout_dq_mask_is_exact(plain_workspace):
    """With K the identity (Nk = d = 128), every value and every dO row equal
    to unit vector 0: dP = dO V^T = 1, D_i = sum_j Pd_ij, and dQ[i, j] =
    scale P_ij (Z_ij / (1 - p) - D_i), positive exactly where Z_ij = 1. Once
    with the bits the dK/dV pass hands on, once drawn in the dQ pass itself."""
    seed, offset, p = 2024, 0, 0.3
    q, _, _, _ = make_qkv_do(1, 2, 300, 128, seed=12, dtype=torch.float32)
    q = (0.2 * q).to(torch.bfloat16)
    k = torch.eye(128).expand(1, 2, 128, 128).contiguous().to(torch.bfloat16)
    v = torch.zeros(1, 2, 128, 128)
    v[..., 0] = 1.0
    dO = torch.zeros(1, 2, 300, 128)
    dO[..., 0] = 1.0
    v, dO = v.to(torch.bfloat16), dO.to(torch.bfloat16)
    got = _run_drop(q, k, v, dO, 1.0 / math.sqrt(128), False, seed, offset, p, plain_workspace)
    want = _mask(seed, offset, p, 1, 2, 300, 128, False)
    assert np.array_equal(got["dq"] > 0, want)
    check("dropout_dq_identity", "bf16", got, _drop_ref(q, k, v, dO, 1.0 / math.sqrt(128), False, seed, offset, p))


@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout_parity(d, causal, p):
    q, k, v, dO = make_qkv_do(1, 2, 300, d, seed=500 + d, dtype=torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    got = _run_drop(q, k, v, dO, scale, causal, 99, 5, p)
    check(f"dropout_d{d}_c{int(causal)}_p{p}", "bf16", got, _drop_ref(q, k, v, dO, scale, causal, 99, 5, p))


def test_dropout_kv_f16_and_d256():
    q, _, _, dO = make_qkv_do(2, 2, 200, 128, seed=5, dtype=torch.float16)
    _, k, v, _ = make_qkv_do(2, 2, 777, 128, seed=6, dtype=torch.float16)
    scale = 1.0 / math.sqrt(128)
    got = _run_drop(q, k, v, dO, scale, True, 123456789, 1, 0.2)
    check("dropout_f16_kv_Nq200_Nk777", "bf16", got, _drop_ref(q, k, v, dO, scale, True, 123456789, 1, 0.2))
    q, k, v, _ = make_qkv_do(1, 2, 333, 256, seed=7, dtype=torch.bfloat16)
    got = _run_drop(q, k, v, None, 1.0 / 16, True, 42, 0, 0.2)
    check("dropout_fwd_d256", "bf16", got, _drop_ref(q, k, v, None, 1.0 / 16, True, 42, 0, 0.2))


def _saved_bits(buf, B, H, Nq, Nk):
    """Unpack a saved-keep-bits buffer into a [B, H, Nq, Nk] bool array (its
    documented layout: per head, query tile and key tile a block of 512
    words, bit 8 (b mod 4) + b // 4 of word w * 128 + r = the bit of row r
    and key 32 w + b)."""
    nqt, nkt = (Nq + 127) // 128, (Nk + 127) // 128
    words = buf.cpu().numpy()[: B * H * nqt * nkt * 2048].view(np.uint32).reshape(B * H, nqt, nkt, 4, 128)
    rows = np.ascontiguousarray(words.transpose(0, 1, 2, 4, 3)).view(np.uint8)  # [BH, qt, kt, row, 16 bytes]
    bits = np.unpackbits(rows, axis=-1, bitorder="little")  # [BH, qt, kt, row, 4 words x 32 bit positions]
    pos = np.array([8 * (b % 4) + b // 4 for b in range(32)])
    bits = bits.reshape(*bits.shape[:-1], 4, 32)[..., pos].reshape(*bits.shape)  # bit positions -> keys
    bits = bits.transpose(0, 1, 3, 2, 4).reshape(B * H, nqt * 128, nkt * 128)[:, :Nq, :Nk]
    return bits.reshape(B, H, Nq, Nk).astype(bool)


@pytest.mark.parametrize("Nq,Nk,causal,p", [(300, 513, False, 0.3), (300, 513, True, 0.3), (128, 128, False, 0.3),
                                            (300, 513, False, 0.7)])
def test_dropout_saved_bits_are_the_oracle_mask(Nq, Nk, causal, p):
    """The forward's saved keep bits equal the oracle's Philox mask bit for
    bit on every visible (query, key) pair (thresholds below and above 128)."""
    import exact_attention_97_gb300 as fa
    seed, offset, B, H = 0xABCDEF0123, 9, 1, 3
    q, _, _, _ = make_qkv_do(B, H, Nq, 64, seed=31, dtype=torch.bfloat16)
    _, k, v, _ = make_qkv_do(B, H, Nk, 64, seed=32, dtype=torch.bfloat16)
    dev = torch.device("cuda")
    mask = fa.dropout_mask_buffer(B, H, Nq, Nk, dev)
    fa.attention_forward(q.to(dev), k.to(dev), v.to(dev), 0.125, causal, dropout_p=p, seed=seed, offset=offset,
                         head_base=5, dropout_mask=mask)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    got = _saved_bits(mask, B, H, Nq, Nk)
    t = oracle.dropout_threshold(p)
    want = np.stack([oracle.dropout_mask(seed, offset, t, 5 + h, Nq, Nk) for h in range(B * H)]).reshape(
        B, H, Nq, Nk).astype(bool)
    visible = np.ones((Nq, Nk), dtype=bool)
    if causal:
        visible = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    assert np.array_equal(got[..., visible], want[..., visible])


@pytest.mark.parametrize("d,Nq,Nk,causal,dtype,p", [(64, 300, 300, True, torch.bfloat16, 0.2),
                                                    (96, 257, 700, True, torch.bfloat16, 0.2),
                                                    (128, 1000, 1000, False, torch.bfloat16, 0.2),
                                                    (128, 200, 777, True, torch.float16, 0.2),
                                                    (128, 513, 300, False, torch.bfloat16, 0.6)])
def test_dropout_saved_bits_give_the_regenerated_results(d, Nq, Nk, causal, dtype, p):
    """Backward from the saved bits equals the backward that draws them again,
    bit for bit (same keep decisions, same arithmetic); both forwards agree too.
    p = 0.6 takes the threshold t >= 128 through every keep-bit path."""
    import exact_attention_97_gb300 as fa
    seed, offset, B, H = 314159, 2, 2, 2
    q, _, _, dO = make_qkv_do(B, H, Nq, d, seed=40 + d, dtype=dtype)
    _, k, v, _ = make_qkv_do(B, H, Nk, d, seed=41 + d, dtype=dtype)
    dev = torch.device("cuda")
    q, k, v, dO = (x.to(dev) for x in (q, k, v, dO))
    scale = 1.0 / math.sqrt(d)
    kw = dict(dropout_p=p, seed=seed, offset=offset)
    o1, l1 = fa.attention_forward(q, k, v, scale, causal, **kw)
    g1 = fa.attention_backward(q, k, v, o1, l1, dO, scale, causal, **kw)
    mask = fa.dropout_mask_buffer(B, H, Nq, Nk, dev)
    o2, l2 = fa.attention_forward(q, k, v, scale, causal, dropout_mask=mask, **kw)
    g2 = fa.attention_backward(q, k, v, o2, l2, dO, scale, causal, dropout_p=p, dropout_mask=mask)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for a, b in zip((o1, l1, *g1), (o2, l2, *g2)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("d,Nq,Nk,causal,dtype,p", [(64, 300, 300, True, torch.bfloat16, 0.2),
                                                    (96, 257, 700, True, torch.bfloat16, 0.2),
                                                    (128, 1000, 1000, False, torch.bfloat16, 0.2),
                                                    (128, 200, 777, True, torch.float16, 0.6),
                                                    (128, 513, 300, False, torch.bfloat16, 0.6)])
def test_dropout_bits_handed_from_dkdv_to_dq(d, Nq, Nk, causal, dtype, p):
    """Given a workspace with room for the keep bits, the dropout backward's
    dK/dV pass writes the bits it draws there and its dQ pass reads them: the
    gradients equal, bit for bit, those of the backward whose passes both
    draw, and the bits left in the workspace are the forward's saved ones on
    every visible (query, key) pair."""
    import exact_attention_97_gb300 as fa
    seed, offset, head_base, B, H = 271828, 4, 3, 2, 2
    q, _, _, dO = make_qkv_do(B, H, Nq, d, seed=50 + d, dtype=dtype)
    _, k, v, _ = make_qkv_do(B, H, Nk, d, seed=51 + d, dtype=dtype)
    dev = torch.device("cuda")
    q, k, v, dO = (x.to(dev) for x in (q, k, v, dO))
    scale = 1.0 / math.sqrt(d)
    kw = dict(dropout_p=p, seed=seed, offset=offset, head_base=head_base)
    kind = fa.FA_F16 if dtype == torch.float16 else fa.FA_BF16
    mask = fa.dropout_mask_buffer(B, H, Nq, Nk, dev)
    o, lse = fa.attention_forward(q, k, v, scale, causal, dropout_mask=mask, **kw)
    plain = torch.empty(fa.fa_bwd_workspace_size(B, H, Nq, d, kind), device=dev, dtype=torch.uint8)
    shared = torch.zeros(fa.fa_bwd_dropout_workspace_size(B, H, Nq, Nk, d, kind), device=dev, dtype=torch.uint8)
    g_drawn = fa.attention_backward(q, k, v, o, lse, dO, scale, causal, workspace=plain, **kw)
    g_handed = fa.attention_backward(q, k, v, o, lse, dO, scale, causal, workspace=shared, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for a, b in zip(g_drawn, g_handed):
        assert torch.equal(a, b)
    got = _saved_bits(shared[plain.numel():], B, H, Nq, Nk)  # the bits follow the plain workspace
    want = _saved_bits(mask, B, H, Nq, Nk)
    visible = np.ones((Nq, Nk), dtype=bool)
    if causal:
        visible = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    assert np.array_equal(got[..., visible], want[..., visible])


def test_dropout_bits_handed_at_full_size():
    """The same at B8 H32 N4096 d128 (32 x 32 blocks per head, every one
    visited): the gradients with and without the handoff are bit-identical,
    and the workspace's bits are byte for byte the forward's saved ones."""
    import exact_attention_97_gb300 as fa
    B, H, N, d, p = 8, 32, 4096, 128, 0.1
    kw = dict(dropout_p=p, seed=0x5151, offset=6)
    dev = torch.device("cuda")
    q, k, v, dO = (x.to(dev) for x in make_qkv_do(B, H, N, d, seed=77, dtype=torch.bfloat16))
    scale = 1.0 / math.sqrt(d)
    mask = fa.dropout_mask_buffer(B, H, N, N, dev)
    o, lse = fa.attention_forward(q, k, v, scale, False, dropout_mask=mask, **kw)
    plain = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d, fa.FA_BF16), device=dev, dtype=torch.uint8)
    shared = torch.zeros(fa.fa_bwd_dropout_workspace_size(B, H, N, N, d, fa.FA_BF16), device=dev,
                         dtype=torch.uint8)
    g_drawn = fa.attention_backward(q, k, v, o, lse, dO, scale, False, workspace=plain, **kw)
    g_handed = fa.attention_backward(q, k, v, o, lse, dO, scale, False, workspace=shared, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    for a, b in zip(g_drawn, g_handed):
        assert torch.equal(a, b)
    assert torch.equal(shared[plain.numel():], mask)


def test_dropout_zero_is_the_plain_path():
    import exact_attention_97_gb300 as fa
    q, k, v, dO = (x.cuda() for x in make_qkv_do(1, 2, 260, 128, seed=8, dtype=torch.bfloat16))
    o, lse = fa.attention_forward(q, k, v, None, True)
    od, lsed = fa.attention_forward(q, k, v, None, True, dropout_p=0.0001, seed=3)  # t = round(0.0256) = 0
    assert torch.equal(o, od) and torch.equal(lse, lsed)
    g = fa.attention_backward(q, k, v, o, lse, dO, None, True)
    gd = fa.attention_backward(q, k, v, o, lse, dO, None, True, dropout_p=0.0001, seed=3)
    for a, b in zip(g, gd):
        assert torch.equal(a, b)


# ------------------------------------------------------------ f16 inputs (same kernels, f16 operands)

@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("N", [1, 127, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_f16_small_and_ragged(d, N, causal):
    q, k, v, dO = make_qkv_do(1, 2, N, d, seed=2000 + N + d, dtype=torch.float16)
    scale = 1.0 / math.sqrt(d)
    got = _as_dict(run_gpu(q, k, v, dO, scale, causal))
    check(f"f16_small_N{N}_d{d}_c{int(causal)}", "bf16", got,
          _full_ref(_np(q), _np(k), _np(v), _np(dO), scale, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_f16_B2_H4_N1024_d128_and_large_scores(causal):
    q, k, v, dO = make_qkv_do(2, 4, 1024, 128, seed=31, dtype=torch.float32)
    q = q * 3  # scores several units wide, so the running max moves
    q, k, v, dO = (x.to(torch.float16) for x in (q, k, v, dO))
    scale = 1.0 / math.sqrt(128)
    got = _as_dict(run_gpu(q, k, v, dO, scale, causal))
    check(f"f16_B2_H4_N1024_d128_c{int(causal)}", "bf16", got,
          _full_ref(_np(q), _np(k), _np(v), _np(dO), scale, causal))


# ------------------------------------------------------------ Nq queries against Nk keys

def _run_gpu_kv(q, k, v, dO, scale, causal):
    import exact_attention_97_gb300 as fa
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, dO))
    nan = float("nan")
    o = torch.full_like(qd, nan)
    lse = torch.full(tuple(q.shape[:3]), nan, device=dev, dtype=torch.float32)
    fa.attention_forward(qd, kd, vd, scale, causal, out=o, lse=lse)
    grads = (torch.full_like(qd, nan), torch.full_like(kd, nan), torch.full_like(vd, nan))
    fa.attention_backward(qd, kd, vd, o, lse, dod, scale, causal, grads=grads)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return dict(zip(("o", "lse", "dq", "dk", "dv"), (t.float().cpu().double().numpy() for t in (o, lse, *grads))))


@pytest.mark.parametrize("Nq,Nk,causal", [(1, 300, True), (1, 300, False), (128, 1000, True), (100, 640, True),
                                          (257, 511, True), (300, 130, False), (640, 641, True)])
@pytest.mark.parametrize("d", [64, 96, 128])
def test_bf16_kv_lengths(Nq, Nk, causal, d):
    """Decode / chunked-prefill shapes: causal mask aligned bottom-right."""
    q, _, _, dO = make_qkv_do(1, 2, Nq, d, seed=300 + Nq, dtype=torch.bfloat16)
    _, k, v, _ = make_qkv_do(1, 2, Nk, d, seed=400 + Nk, dtype=torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    got = _run_gpu_kv(q, k, v, dO, scale, causal)
    o, lse = oracle.attention_fwd_kv(_np(q), _np(k), _np(v), scale, causal)
    dq, dk, dv = oracle.attention_bwd_kv(_np(q), _np(k), _np(v), _np(dO), scale, causal)
    check(f"bf16_kv_Nq{Nq}_Nk{Nk}_d{d}_c{int(causal)}", "bf16", got,
          {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv})


def test_f16_kv_lengths():
    q, _, _, dO = make_qkv_do(2, 2, 200, 128, seed=5, dtype=torch.float16)
    _, k, v, _ = make_qkv_do(2, 2, 777, 128, seed=6, dtype=torch.float16)
    scale = 1.0 / math.sqrt(128)
    got = _run_gpu_kv(q, k, v, dO, scale, True)
    o, lse = oracle.attention_fwd_kv(_np(q), _np(k), _np(v), scale, True)
    dq, dk, dv = oracle.attention_bwd_kv(_np(q), _np(k), _np(v), _np(dO), scale, True)
    check("f16_kv_Nq200_Nk777_d128_c1", "bf16", got, {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv})


def test_bf16_causal_B1_H8_N1024_d64():
    w = WORKLOADS["bf16_causal_B1_H8_N1024_d64"]
    q, k, v, dO = make_qkv_do(w.B, w.H, w.N, w.d, w.seed, torch.bfloat16)
    got = _as_dict(run_gpu(q, k, v, dO, w.scale, w.causal))
    check(w.name, "bf16", got, _full_ref(_np(q), _np(k), _np(v), _np(dO), w.scale, w.causal))


# ------------------------------------------------------------ full-size workloads, sampled

def _head_ref(q, k, v, dO, b, h, scale, causal, rows=None, keys=None):
    """Oracle for one head: O, L, dQ at `rows` and dK, dV at `keys` (all if None)."""
    N = q.shape[2]
    qh, kh, vh, doh = (_np(x[b, h]) for x in (q, k, v, dO))
    rows = np.arange(N) if rows is None else np.asarray(rows)
    keys = np.arange(N) if keys is None else np.asarray(keys)
    o, lse, dq = oracle.query_rows(qh, kh, vh, doh, rows, scale, causal)
    dk, dv = oracle.key_rows(qh, kh, vh, doh, keys, scale, causal)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, rows, keys


def _sampled_check(name, w, q, k, v, dO, got, heads, n_rows=64):
    B, H, N = w.B, w.H, w.N
    # whole heads
    for (b, h) in heads:
        ref, rows, keys = _head_ref(q, k, v, dO, b, h, w.scale, w.causal)
        g = {"o": got["o"][b, h], "lse": got["lse"][b, h], "dq": got["dq"][b, h],
             "dk": got["dk"][b, h], "dv": got["dv"][b, h]}
        check(f"{name}_head{b}_{h}", "bf16", g, ref)
    # seeded query rows spread over all heads
    flat = sample_indices(B * H * N, n_rows, seed=99).numpy()
    o_r, l_r, dq_r = [], [], []
    for idx in flat:
        b, h, i = idx // (H * N), (idx // N) % H, idx % N
        ref, _, _ = _head_ref(q, k, v, dO, b, h, w.scale, w.causal, rows=[i], keys=[])
        o_r.append((got["o"][b, h, i], ref["o"][0]))
        l_r.append((got["lse"][b, h, i], ref["lse"][0]))
        dq_r.append((got["dq"][b, h, i], ref["dq"][0]))
    g = {"o": np.array([a for a, _ in o_r]), "lse": np.array([a for a, _ in l_r]),
         "dq": np.array([a for a, _ in dq_r])}
    r = {"o": np.array([b for _, b in o_r]), "lse": np.array([b for _, b in l_r]),
         "dq": np.array([b for _, b in dq_r])}
    check(f"{name}_rows", "bf16", g, r)


def test_bf16_B4_H16_N4096_d64():
    w = WORKLOADS["bf16_B4_H16_N4096_d64"]
    q, k, v, dO = make_qkv_do(w.B, w.H, w.N, w.d, w.seed, torch.bfloat16)
    got = _as_dict(run_gpu(q, k, v, dO, w.scale, w.causal))
    _sampled_check(w.name, w, q, k, v, dO, got, heads=[(0, 0), (3, 15)])


def test_bf16_B8_H32_N4096_d128():
    w = WORKLOADS["bf16_B8_H32_N4096_d128"]
    q, k, v, dO = make_qkv_do(w.B, w.H, w.N, w.d, w.seed, torch.bfloat16)
    got = _as_dict(run_gpu(q, k, v, dO, w.scale, w.causal))
    _sampled_check(w.name, w, q, k, v, dO, got, heads=[(0, 0), (7, 31)])


def test_bf16_causal_B1_H32_N65536_d128():
    w = WORKLOADS["bf16_causal_B1_H32_N65536_d128"]
    q, k, v, dO = make_qkv_do(w.B, w.H, w.N, w.d, w.seed, torch.bfloat16)
    got = _as_dict(run_gpu(q, k, v, dO, w.scale, w.causal))
    N = w.N
    # 256 seeded query rows over all heads: O, L, dQ (each row costs O(N d))
    flat = sample_indices(w.H * N, 256, seed=5).numpy()
    by_head = {}
    for idx in flat:
        by_head.setdefault(int(idx // N), []).append(int(idx % N))
    g, r = {"o": [], "lse": [], "dq": []}, {"o": [], "lse": [], "dq": []}
    for h, rows in by_head.items():
        qh, kh, vh, doh = (_np(x[0, h]) for x in (q, k, v, dO))
        o, lse, dq = oracle.query_rows(qh, kh, vh, doh, rows, w.scale, True)
        g["o"].append(got["o"][0, h, rows]); r["o"].append(o)
        g["lse"].append(got["lse"][0, h, rows]); r["lse"].append(lse)
        g["dq"].append(got["dq"][0, h, rows]); r["dq"].append(dq)
    check(w.name + "_rows", "bf16", {k_: np.concatenate(v_) for k_, v_ in g.items()},
          {k_: np.concatenate(v_) for k_, v_ in r.items()})
    # 256 key rows: 64 seeded keys in the last 4096 positions of 4 heads (a key's
    # gradient needs every later query's L and D, so late keys keep this bounded)
    gk, rk = {"dk": [], "dv": []}, {"dk": [], "dv": []}
    for h in (0, 9, 22, 31):
        keys = (N - 4096 + sample_indices(4096, 64, seed=h).numpy()).tolist()
        qh, kh, vh, doh = (_np(x[0, h]) for x in (q, k, v, dO))
        dk, dv = oracle.key_rows(qh, kh, vh, doh, keys, w.scale, True)
        gk["dk"].append(got["dk"][0, h, keys]); rk["dk"].append(dk)
        gk["dv"].append(got["dv"][0, h, keys]); rk["dv"].append(dv)
    check(w.name + "_keys", "bf16", {k_: np.concatenate(v_) for k_, v_ in gk.items()},
          {k_: np.concatenate(v_) for k_, v_ in rk.items()})
    # two whole heads: every key's dK and dV (and every row's dQ) against the
    # full fp64 backward of the head. Early keys sum the contributions of up
    # to 512 query tiles in the dK/dV pass's accumulators.
    for h in (int(x) for x in sample_indices(w.H, 2, seed=65536).numpy()):
        qh, kh, vh, doh = (_np(x[:, h:h + 1]) for x in (q, k, v, dO))
        rdq, rdk, rdv = oracle.attention_bwd(qh, kh, vh, doh, w.scale, True)
        check(f"{w.name}_whole_head{h}", "bf16",
              {"dq": got["dq"][:, h:h + 1], "dk": got["dk"][:, h:h + 1], "dv": got["dv"][:, h:h + 1]},
              {"dq": rdq, "dk": rdk, "dv": rdv})
        # the earliest keys carry the longest sums: hold their block to the same bar
        check(f"{w.name}_whole_head{h}_first_block", "bf16",
              {"dk": got["dk"][0, h, :128], "dv": got["dv"][0, h, :128]},
              {"dk": rdk[0, 0, :128], "dv": rdv[0, 0, :128]})
    # any-size properties over every key of every head: rows of P sum to one, so
    # sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i
    dk_sum = got["dk"].sum(axis=2)
    dv_sum = got["dv"].sum(axis=2)
    do_sum = _np(dO).sum(axis=2)
    assert np.max(np.abs(dk_sum)) <= 1e-2 * np.max(np.abs(got["dk"]).sum(axis=2))
    assert np.max(np.abs(dv_sum - do_sum)) <= 1e-2 * np.max(np.abs(got["dv"]).sum(axis=2))


def test_repeated_calls_are_stable():
    """The same call twice gives the same O and L (no state leaks between calls)."""
    q, k, v, dO = make_qkv_do(2, 3, 333, 128, seed=3, dtype=torch.bfloat16)
    a = run_gpu(q, k, v, dO, 0.1, True, backward=False)
    b = run_gpu(q, k, v, dO, 0.1, True, backward=False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
