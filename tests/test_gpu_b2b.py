"""GPU parity: fused B2BGEMM (cf_b2bgemm through the C ABI) against the
float64 oracle, on the attention shape (S = Q K^T, F = scaled softmax or
scaled ReLU, O = bf16(F(S)) V) and the MLP shape (ReLU)."""
import math

import numpy as np
import pytest
import torch

from oracle import cf_oracle as O
from back_gemm_fusion_gb300 import inputs as I
from tests.parity import sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from back_gemm_fusion_gb300 import build
    build.build()
    import back_gemm_fusion_gb300 as cf
    return cf


def b2b_gate(gpu, ref, absbound, what):
    """Contract gate plus a per-element bound derived from the single bf16
    rounding of the intermediate: each element of S' may differ by one bf16
    ulp (2^-8 relative) between the GPU (fp32 S') and the oracle (fp64 S'),
    so |dO| <= 2^-7 (|S'| . |W2|) covers it with a factor-2 margin (the
    online-softmax form rounds exp(s - m) before dividing by l)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))
    assert np.all(err <= 1e-2 * np.maximum(1.0, rms)), f"{what}: contract gate, max err {err.max():.3g}"
    bound = 2.0 ** -7 * absbound + 1e-5 * rms + 1e-7
    worst = (err / bound).max()
    assert worst <= 1.0, f"{what}: bf16-derived bound exceeded ({worst:.3g} x)"


def _abs_bound(q, k, v, op, scale):
    """|S'| . |W2| with S' = F(scale q k^T) unrounded (float64)."""
    S = q @ k.T
    return np.abs(O.mid_op(S, op, scale)) @ np.abs(v)


def _attention_case(batch, L, op, seed, growth=None):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((batch, L, 128))
    k = rng.standard_normal((batch, L, 128))
    if growth is not None:  # make later key blocks dominate: forces online rescaling
        k = k * (1.0 + growth * (np.arange(L) // 128))[None, :, None]
    v = rng.standard_normal((batch, L, 128))
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    return t(q), t(k), t(v)


def _run_attention(cf, Q, K, V, op, scale, key_split=0):
    out = cf.cf_b2bgemm(Q.cuda(), K.cuda(), V.cuda(), op, scale, w1_trans=True, key_split=key_split)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    return out.cpu().numpy()


# key_split: 1 = one CTA walks all keys of a query block (the online C = 1
# form); 2 = two CTAs of a cluster split each block's keys (for these short
# key ranges AUTO keeps one CTA: too few chunks to pay for the merge).
@pytest.mark.parametrize("key_split", [1, 2])
@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
@pytest.mark.parametrize("batch,L", [(1, 128), (2, 256), (3, 384), (2, 1024)])
def test_attention_small(cf, batch, L, op, key_split):
    Q, K, V = _attention_case(batch, L, op, seed=L + batch)
    scale = 1 / math.sqrt(128)
    got = _run_attention(cf, Q, K, V, op, scale, key_split)
    q, k, v = (I.to_f64(t) for t in (Q, K, V))
    for b in range(batch):
        ref = O.b2bgemm(q[b], k[b].T, v[b], op, scale)
        b2b_gate(got[b], ref, _abs_bound(q[b], k[b], v[b], op, scale), f"attention {op} b={b} L={L}")


@pytest.mark.parametrize("key_split", [1, 4])
@pytest.mark.parametrize("growth", [2.0, 6.0])
def test_attention_softmax_rescales(cf, growth, key_split):
    # Logits grow block by block, so the running max increases by more than
    # 2^8 in exp2 units several times: exercises the O rescale path.  With
    # the key split each CTA rescales on its own range and the merge meets
    # maxima that differ by far more than 2^8 between the CTAs.
    Q, K, V = _attention_case(2, 1024, "scale_softmax", seed=11, growth=growth)
    scale = 1 / math.sqrt(128)
    got = _run_attention(cf, Q, K, V, "scale_softmax", scale, key_split)
    q, k, v = (I.to_f64(t) for t in (Q, K, V))
    for b in range(2):
        ref = O.b2bgemm(q[b], k[b].T, v[b], "scale_softmax", scale)
        b2b_gate(got[b], ref, _abs_bound(q[b], k[b], v[b], "scale_softmax", scale), f"rescale b={b}")


@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
def test_attention_full_size_sampled(cf, op):
    case = I.attention_b2b(op=op)
    got = _run_attention(cf, case.A, case.W1, case.W2, op, case.scale)
    rng = np.random.default_rng(1)
    heads = rng.choice(case.batch, size=8, replace=False)
    for h in heads:
        rows = sample_rows(case.M, 32, seed=int(h))
        q = I.to_f64(case.A[h])
        k = I.to_f64(case.W1[h])
        v = I.to_f64(case.W2[h])
        ref = O.b2bgemm(q[rows], k.T, v, op, case.scale)
        b2b_gate(got[h][rows], ref, _abs_bound(q[rows], k, v, op, case.scale), f"attention {op} head {h}")


@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
@pytest.mark.parametrize("Lq", [1, 77, 200])
def test_attention_ragged_queries(cf, Lq, op):
    # Fewer (or not a multiple of 128) query rows than keys: the last query
    # block is zero-filled on load and its rows past Lq are not stored.
    rng = np.random.default_rng(Lq)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    Q = t(rng.standard_normal((2, Lq, 128)))
    K = t(rng.standard_normal((2, 256, 128)))
    V = t(rng.standard_normal((2, 256, 128)))
    scale = 1 / math.sqrt(128)
    got = _run_attention(cf, Q, K, V, op, scale)
    assert got.shape == (2, Lq, 128)
    q, k, v = (I.to_f64(x) for x in (Q, K, V))
    for b in range(2):
        ref = O.b2bgemm(q[b], k[b].T, v[b], op, scale)
        b2b_gate(got[b], ref, _abs_bound(q[b], k[b], v[b], op, scale), f"attention {op} Lq={Lq} b={b}")


def test_attention_zero_keys_column_mean(cf):
    # Q K^T == 0 -> P = 1/L exactly -> O = column mean of V (closed form).
    L = 2048
    Q, _, V = _attention_case(1, L, "scale_softmax", seed=3)
    K = torch.zeros_like(Q)
    got = _run_attention(cf, Q, K, V, "scale_softmax", 1 / math.sqrt(128))
    mean = I.to_f64(V)[0].mean(axis=0)
    np.testing.assert_allclose(got[0], np.broadcast_to(mean, (L, 128)), rtol=0, atol=2e-6)


# ------------------------------------------------------------------ MLP shape
def _mlp_case(M, K, N1, N2, seed):
    rng = np.random.default_rng(seed)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    X = t(rng.standard_normal((M, K)))
    W1 = t(rng.standard_normal((K, N1)) / math.sqrt(K))
    W2 = t(rng.standard_normal((N1, N2)) / math.sqrt(N1))
    return X, W1, W2


@pytest.mark.parametrize("w1_trans", [False, True])
@pytest.mark.parametrize("op,scale", [("relu", 1.0), ("scale_relu", 0.75)])
@pytest.mark.parametrize("M,K,N1,N2", [(128, 64, 128, 256), (256, 128, 512, 256), (384, 192, 1024, 512),
                                       (256, 256, 1024, 1024), (128, 64, 512, 1024), (512, 192, 1024, 512),
                                       (768, 64, 2048, 1024)])
def test_mlp_small(cf, M, K, N1, N2, op, scale, w1_trans):
    X, W1, W2 = _mlp_case(M, K, N1, N2, seed=M + K + N1 + N2)
    W1d = W1.t().contiguous().cuda() if w1_trans else W1.cuda()
    out = cf.cf_b2bgemm(X.cuda(), W1d, W2.cuda(), op, scale, w1_trans=w1_trans)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    x, w1, w2 = (I.to_f64(t) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, op, scale)
    bound = np.abs(O.mid_op(x @ w1, op, scale)) @ np.abs(w2)
    b2b_gate(out.cpu().numpy(), ref, bound, f"mlp {op} {M}x{K}x{N1}x{N2} trans={w1_trans}")


@pytest.mark.parametrize("w1_trans", [False, True])
@pytest.mark.parametrize("M,K,N1,N2", [(1, 512, 128, 256), (8, 512, 128, 256), (64, 512, 128, 256),
                                       (77, 200, 512, 256), (300, 72, 1024, 1024)])
def test_mlp_ragged(cf, M, K, N1, N2, w1_trans):
    # Ragged M (the last 128-row strip is partial: zero-filled loads, rows
    # past M not stored) and K not a multiple of 64 (the last K block reads
    # zeros); the first three are the bottom-MLP shape 512 -> 128 -> 256 at
    # batch 1, 8 and 64.
    X, W1, W2 = _mlp_case(M, K, N1, N2, seed=M * 7 + K)
    W1d = W1.t().contiguous().cuda() if w1_trans else W1.cuda()
    out = cf.cf_b2bgemm(X.cuda(), W1d, W2.cuda(), "relu", 1.0, w1_trans=w1_trans)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    x, w1, w2 = (I.to_f64(t) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, "relu", 1.0)
    bound = np.abs(O.mid_op(x @ w1, "relu", 1.0)) @ np.abs(w2)
    b2b_gate(out.cpu().numpy(), ref, bound, f"mlp ragged {M}x{K}x{N1}x{N2} trans={w1_trans}")


@pytest.mark.parametrize("M,K,N1,N2,w1_trans", [(64, 16, 512, 256, False), (300, 8, 256, 1024, True),
                                                (129, 56, 384, 600, False), (1, 24, 128, 512, True)])
def test_mlp_short_k(cf, M, K, N1, N2, w1_trans):
    # K below one 64-wide block (a first layer over a few dense features,
    # 13 padded to 16): the only K block of X and W1 reads zeros past K.
    X, W1, W2 = _mlp_case(M, K, N1, N2, seed=M * 11 + K)
    W1d = W1.t().contiguous().cuda() if w1_trans else W1.cuda()
    out = cf.cf_b2bgemm(X.cuda(), W1d, W2.cuda(), "relu", 1.0, w1_trans=w1_trans)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    x, w1, w2 = (I.to_f64(t) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, "relu", 1.0)
    bound = np.abs(O.mid_op(x @ w1, "relu", 1.0)) @ np.abs(w2)
    b2b_gate(out.cpu().numpy(), ref, bound, f"mlp short K {M}x{K}x{N1}x{N2} trans={w1_trans}")


@pytest.mark.parametrize("batch,M,K,N1,N2,w1_trans", [(1, 384, 128, 640, 600, False), (2, 257, 64, 384, 1024, True),
                                                       (3, 512, 96, 256, 256, False)])
def test_mlp_batched(cf, batch, M, K, N1, N2, w1_trans):
    # Batch entries (strided A, W1, W2 and output), three CTAs per cluster
    # (N2 = 600), and a last 128-row strip holding one row (M = 257).
    rng = np.random.default_rng(batch * 1000 + M)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    X = t(rng.standard_normal((batch, M, K)))
    W1 = t(rng.standard_normal((batch, K, N1)) / math.sqrt(K))
    W2 = t(rng.standard_normal((batch, N1, N2)) / math.sqrt(N1))
    W1d = W1.transpose(1, 2).contiguous().cuda() if w1_trans else W1.cuda()
    out = cf.cf_b2bgemm(X.cuda(), W1d, W2.cuda(), "relu", w1_trans=w1_trans)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    got = out.cpu().numpy()
    for b in range(batch):
        x, w1, w2 = (I.to_f64(a[b]) for a in (X, W1, W2))
        ref = O.b2bgemm(x, w1, w2, "relu")
        bound = np.abs(O.mid_op(x @ w1, "relu")) @ np.abs(w2)
        b2b_gate(got[b], ref, bound, f"mlp batch {b} {M}x{K}x{N1}x{N2}")


def test_mlp_full_size_sampled(cf):
    case = I.mlp_b2b()
    out = cf.cf_b2bgemm(case.A[0].cuda(), case.W1[0].cuda(), case.W2[0].cuda(), "relu")
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    rows = sample_rows(case.M)
    x, w1, w2 = I.to_f64(case.A[0])[rows], I.to_f64(case.W1[0]), I.to_f64(case.W2[0])
    ref = O.b2bgemm(x, w1, w2, "relu")
    bound = np.abs(O.mid_op(x @ w1, "relu")) @ np.abs(w2)
    b2b_gate(out.cpu().numpy()[rows], ref, bound, "mlp 16384x1024x4096x1024")


def test_b2b_rejects_unsupported(cf):
    X, W1, W2 = _mlp_case(128, 64, 384, 1280, seed=1)  # N2 = 1280: five CTAs per cluster
    with pytest.raises(cf.CFError):
        cf.cf_b2bgemm(X.cuda(), W1.cuda(), W2.cuda(), "relu")
    X, W1, W2 = _mlp_case(128, 64, 384, 256, seed=1)   # softmax on the MLP shape (W1 not transposed)
    with pytest.raises(cf.CFError):
        cf.cf_b2bgemm(X.cuda(), W1.cuda(), W2.cuda(), "scale_softmax", 0.5)
    Q = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cf.CFError):                     # softmax with a non-positive scale
        cf.cf_b2bgemm(Q, Q, Q, "scale_softmax", -1.0, w1_trans=True)


def _bf16_gate(gpu, ref, absbound, what):
    """bf16 output: the fp32 result (within the B2B bound of the oracle) is
    rounded once more to nearest even (unit roundoff 2^-8), which adds
    2^-8 |ref| (plus its own
    small share of the fp32 bound).  The fp32 contract gate is taken on the
    fp32 output of the same call; a bf16 value of magnitude 2^k carries a
    half-ulp of 2^(k-8), more than 1e-2 rms for large elements."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))
    bound = (2.0 ** -7 * absbound + 1e-5 * rms + 1e-7) * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref)
    worst = (np.abs(gpu - ref) / bound).max()
    assert worst <= 1.0, f"{what}: bf16-output bound exceeded ({worst:.3g} x)"


@pytest.mark.parametrize("key_split", [1, 2])
@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
@pytest.mark.parametrize("batch,Lq,L", [(2, 256, 256), (2, 77, 384), (1, 128, 1024)])
def test_attention_bf16_output(cf, batch, Lq, L, op, key_split):
    rng = np.random.default_rng(Lq + L)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    Q, K, V = (t(rng.standard_normal((batch, n, 128))) for n in (Lq, L, L))
    scale = 1 / math.sqrt(128)
    g = cf.cf_b2bgemm(Q.cuda(), K.cuda(), V.cuda(), op, scale, w1_trans=True, out_dtype=torch.bfloat16,
                      key_split=key_split)
    f = cf.cf_b2bgemm(Q.cuda(), K.cuda(), V.cuda(), op, scale, w1_trans=True, key_split=key_split)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    assert g.dtype == torch.bfloat16 and g.shape == (batch, Lq, 128)
    assert torch.equal(g.cpu(), f.cpu().to(torch.bfloat16)), "bf16 out differs from the rounded fp32 out"
    q, k, v = (I.to_f64(x) for x in (Q, K, V))
    got = g.float().cpu().numpy()
    got32 = f.cpu().numpy()
    for b in range(batch):
        ref = O.b2bgemm(q[b], k[b].T, v[b], op, scale)
        bound = _abs_bound(q[b], k[b], v[b], op, scale)
        b2b_gate(got32[b], ref, bound, f"attention fp32 {op} b={b}")
        _bf16_gate(got[b], ref, bound, f"attention bf16 {op} b={b}")


@pytest.mark.parametrize("M,K,N1,N2", [(77, 200, 512, 256), (256, 128, 1024, 1024), (8, 512, 128, 256)])
def test_mlp_bf16_output(cf, M, K, N1, N2):
    X, W1, W2 = _mlp_case(M, K, N1, N2, seed=M + 3 * K)
    g = cf.cf_b2bgemm(X.cuda(), W1.cuda(), W2.cuda(), "relu", out_dtype=torch.bfloat16)
    f = cf.cf_b2bgemm(X.cuda(), W1.cuda(), W2.cuda(), "relu")
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    assert torch.equal(g.cpu(), f.cpu().to(torch.bfloat16)), "bf16 out differs from the rounded fp32 out"
    x, w1, w2 = (I.to_f64(t) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, "relu")
    bound = np.abs(O.mid_op(x @ w1, "relu")) @ np.abs(w2)
    b2b_gate(f.cpu().numpy(), ref, bound, f"mlp fp32 {M}x{K}x{N1}x{N2}")
    _bf16_gate(g.float().cpu().numpy(), ref, bound, f"mlp bf16 {M}x{K}x{N1}x{N2}")


def _bf16_t(a):
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("key_split", [1, 2])
@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
@pytest.mark.parametrize("Lq,N1", [(128, 1), (200, 77), (256, 200), (128, 1000)])
def test_attention_ragged_keys(cf, Lq, N1, op, key_split):
    # N1 not a multiple of the 128-key chunk: the last chunk's keys past N1
    # load as zero rows and leave the softmax max and sum; V rows past N1
    # are zero (target-attention-like short key sequences).
    rng = np.random.default_rng(N1 + Lq)
    Q = _bf16_t(rng.standard_normal((2, Lq, 128)))
    K = _bf16_t(rng.standard_normal((2, N1, 128)))
    V = _bf16_t(rng.standard_normal((2, N1, 128)))
    scale = 1 / math.sqrt(128)
    got = _run_attention(cf, Q, K, V, op, scale, key_split)
    q, k, v = (I.to_f64(x) for x in (Q, K, V))
    for b in range(2):
        ref = O.b2bgemm(q[b], k[b].T, v[b], op, scale)
        b2b_gate(got[b], ref, _abs_bound(q[b], k[b], v[b], op, scale), f"attention {op} Lq={Lq} N1={N1} b={b}")


@pytest.mark.parametrize("key_split", [1, 2])
@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
@pytest.mark.parametrize("d_qk,d_v,N1", [(64, 64, 256), (64, 64, 200), (128, 64, 384), (96, 32, 130),
                                         (32, 128, 512)])
def test_attention_head_dims(cf, d_qk, d_v, N1, op, key_split):
    # Head dims below 128: Q/K columns past d_qk and V columns past d_v load
    # as zeros; the output has d_v columns.
    rng = np.random.default_rng(d_qk * 7 + d_v + N1)
    Lq = 200
    Q = _bf16_t(rng.standard_normal((2, Lq, d_qk)))
    K = _bf16_t(rng.standard_normal((2, N1, d_qk)))
    V = _bf16_t(rng.standard_normal((2, N1, d_v)))
    scale = 1 / math.sqrt(d_qk)
    out = cf.cf_b2bgemm(Q.cuda(), K.cuda(), V.cuda(), op, scale, w1_trans=True, key_split=key_split)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    assert out.shape == (2, Lq, d_v)
    got = out.cpu().numpy()
    q, k, v = (I.to_f64(x) for x in (Q, K, V))
    for b in range(2):
        ref = O.b2bgemm(q[b], k[b].T, v[b], op, scale)
        b2b_gate(got[b], ref, _abs_bound(q[b], k[b], v[b], op, scale), f"attention {op} d={d_qk}/{d_v} b={b}")


@pytest.mark.parametrize("M,K,N1,N2", [(256, 128, 200, 256), (200, 64, 1000, 296), (128, 256, 384, 1000),
                                       (64, 512, 104, 520), (300, 72, 136, 8)])
def test_mlp_ragged_n(cf, M, K, N1, N2):
    # N1 not a multiple of 128 C (chunks past N1 are zero) and N2 not a
    # multiple of 256 (the last CTA's output block is clipped).
    X, W1, W2 = _mlp_case(M, K, N1, N2, seed=M + N1 + N2)
    out = cf.cf_b2bgemm(X.cuda(), W1.cuda(), W2.cuda(), "relu")
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    x, w1, w2 = (I.to_f64(t) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, "relu")
    bound = np.abs(O.mid_op(x @ w1, "relu")) @ np.abs(w2)
    b2b_gate(out.cpu().numpy(), ref, bound, f"mlp ragged N {M}x{K}x{N1}x{N2}")


def test_mlp_ragged_n2_bf16_padded(cf):
    # bf16 output of 296 columns inside 304-element rows: the padding stays.
    X, W1, W2 = _mlp_case(256, 128, 256, 296, seed=3)
    buf = torch.full((256, 304), 3.0, dtype=torch.bfloat16, device="cuda")
    cf.cf_b2bgemm(X.cuda(), W1.cuda(), W2.cuda(), "relu", out=buf[:, :296])
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    assert torch.all(buf[:, 296:] == 3.0)
    x, w1, w2 = (I.to_f64(t) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, "relu")
    bound = np.abs(O.mid_op(x @ w1, "relu")) @ np.abs(w2)
    _bf16_gate(buf[:, :296].float().cpu().numpy(), ref, bound, "mlp N2=296 bf16")


@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
def test_target_attention_shape(cf, op):
    # The target-attention bench shape (512 targets over 200 behaviours,
    # d = 128) at batch 4, every row compared.
    case = I.target_attention(batch=4, op=op)
    got = _run_attention(cf, case.A, case.W1, case.W2, op, case.scale)
    for b in range(case.batch):
        q, k, v = (I.to_f64(t[b]) for t in (case.A, case.W1, case.W2))
        ref = O.b2bgemm(q, k.T, v, op, case.scale)
        b2b_gate(got[b], ref, _abs_bound(q, k, v, op, case.scale), f"target attention {op} b={b}")


# ------------------------------------------------------------ key split (Eq. 5)
@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
@pytest.mark.parametrize("key_split", [2, 3, 5, 8, 0])
def test_attention_key_split(cf, key_split, op):
    # One query block over 2048 keys (16 chunks) split across a cluster:
    # 3 CTAs take 6 + 6 + 4 chunks, a request of 5 becomes 4 CTAs of 4
    # chunks, 8 CTAs take 2 each, and AUTO picks 2 (at least 8 chunks per
    # CTA).  The merged (m, l, O) must match the oracle like the one-CTA
    # form does.
    Q, K, V = _attention_case(2, 2048, op, seed=40 + key_split)
    Q = Q[:, :128].contiguous()
    scale = 1 / math.sqrt(128)
    got = _run_attention(cf, Q, K, V, op, scale, key_split)
    q, k, v = (I.to_f64(x) for x in (Q, K, V))
    for b in range(2):
        ref = O.b2bgemm(q[b], k[b].T, v[b], op, scale)
        b2b_gate(got[b], ref, _abs_bound(q[b], k[b], v[b], op, scale), f"key split {key_split} {op} b={b}")


@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
def test_attention_key_split_decode_shape(cf, op):
    # Few query rows over a long key sequence (4 heads x 77 queries x 8192
    # keys, ragged query block): AUTO splits each block over 8 CTAs.
    rng = np.random.default_rng(5)
    Q = _bf16_t(rng.standard_normal((4, 77, 128)))
    K = _bf16_t(rng.standard_normal((4, 8192, 128)))
    V = _bf16_t(rng.standard_normal((4, 8192, 128)))
    scale = 1 / math.sqrt(128)
    got = _run_attention(cf, Q, K, V, op, scale, 0)
    one = _run_attention(cf, Q, K, V, op, scale, 1)
    q, k, v = (I.to_f64(x) for x in (Q, K, V))
    for b in range(4):
        ref = O.b2bgemm(q[b], k[b].T, v[b], op, scale)
        bound = _abs_bound(q[b], k[b], v[b], op, scale)
        b2b_gate(got[b], ref, bound, f"decode shape split {op} b={b}")
        b2b_gate(one[b], ref, bound, f"decode shape one CTA {op} b={b}")


def test_attention_key_split_ragged_head_dim_bf16(cf):
    # Split with ragged keys (N1 = 1000: 8 chunks, the last with 104 keys),
    # a value head dim of 30 written into 32-element rows (the last
    # four-column group of each row is partial), fp32 and bf16 outputs.
    rng = np.random.default_rng(6)
    Q = _bf16_t(rng.standard_normal((2, 200, 64)))
    K = _bf16_t(rng.standard_normal((2, 1000, 64)))
    V = _bf16_t(rng.standard_normal((2, 1000, 30)))
    Vp = torch.zeros((2, 1000, 32), dtype=torch.bfloat16, device="cuda")  # 16-byte row pitch
    Vp[:, :, :30] = V.cuda()
    scale = 1 / 8.0
    q, k, v = (I.to_f64(x) for x in (Q, K, V))
    for dt in (torch.float32, torch.bfloat16):
        buf = torch.full((2, 200, 32), 9.0, dtype=dt, device="cuda")
        cf.cf_b2bgemm(Q.cuda(), K.cuda(), Vp[:, :, :30], "scale_softmax", scale, w1_trans=True, out=buf[:, :, :30],
                      key_split=3)
        torch.cuda.synchronize()
        assert cf.cf_last_device_status() == 0
        assert torch.all(buf[:, :, 30:] == 9.0)
        got = buf[:, :, :30].float().cpu().numpy()
        for b in range(2):
            ref = O.b2bgemm(q[b], k[b].T, v[b], "scale_softmax", scale)
            bound = _abs_bound(q[b], k[b], v[b], "scale_softmax", scale)
            if dt == torch.float32:
                b2b_gate(got[b], ref, bound, f"split ragged fp32 b={b}")
            else:
                _bf16_gate(got[b], ref, bound, f"split ragged bf16 b={b}")


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_b2b_output_rows_16_byte_aligned(cf, dt):
    # Output rows that start on 16-byte but not 32-byte boundaries take the
    # 16-byte store path (32-byte aligned rows are written a whole 32-byte
    # sector per store); the padding past each row stays untouched.
    rng = np.random.default_rng(8)
    scale = 1 / math.sqrt(128)
    Q = _bf16_t(rng.standard_normal((2, 200, 128)))
    K = _bf16_t(rng.standard_normal((2, 384, 128)))
    V = _bf16_t(rng.standard_normal((2, 384, 128)))
    pitch = 132 if dt == torch.float32 else 136
    buf = torch.full((2, 200, pitch), 5.0, dtype=dt, device="cuda")
    cf.cf_b2bgemm(Q.cuda(), K.cuda(), V.cuda(), "scale_softmax", scale, w1_trans=True, out=buf[:, :, :128])
    X, W1, W2 = _mlp_case(200, 128, 512, 256, seed=9)
    mpitch = 260 if dt == torch.float32 else 264
    mbuf = torch.full((200, mpitch), 5.0, dtype=dt, device="cuda")
    cf.cf_b2bgemm(X.cuda(), W1.cuda(), W2.cuda(), "relu", out=mbuf[:, :256])
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    assert torch.all(buf[:, :, 128:] == 5.0) and torch.all(mbuf[:, 256:] == 5.0)
    gate = b2b_gate if dt == torch.float32 else _bf16_gate
    q, k, v = (I.to_f64(x) for x in (Q, K, V))
    got = buf[:, :, :128].float().cpu().numpy()
    for b in range(2):
        ref = O.b2bgemm(q[b], k[b].T, v[b], "scale_softmax", scale)
        gate(got[b], ref, _abs_bound(q[b], k[b], v[b], "scale_softmax", scale), f"attention 16-byte rows b={b}")
    x, w1, w2 = (I.to_f64(t) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, "relu")
    gate(mbuf[:, :256].float().cpu().numpy(), ref, np.abs(O.mid_op(x @ w1, "relu")) @ np.abs(w2), "mlp 16-byte rows")
