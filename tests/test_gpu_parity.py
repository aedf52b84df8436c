"""GPU parity: every step of the CUDA path against the fp64 oracle, through the C ABI.

Each stage gets identical inputs on both sides.  Inputs come from the seeded generators
or from the oracle itself (e.g. the prepare stage takes the oracle's Hessian rounded to
fp32; the quantize stage takes the oracle's U rounded to fp32); no oracle input is ever
produced by the CUDA path.
"""

import math

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from post_weight_quantization_03_gb300 import build_lib, gptq
from post_weight_quantization_03_gb300 import synthetic as S
from tests import parity as PT

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    gptq.load()
    torch.cuda.init()


def _x(spec, n_tok=None):
    X = S.activations(spec, device="cpu", n_tok=n_tok)
    return X


def _padded(X, dev=DEV):
    """X on the device with its row pitch rounded up to 16 bytes (an ABI requirement)."""
    n, d = X.shape
    step = 16 // X.element_size()
    ld = (d + step - 1) // step * step
    buf = torch.zeros(n, ld, dtype=X.dtype, device=dev)
    buf[:, :d] = X.to(dev)
    return buf[:, :d]


def _codes(qpacked, bits, d):
    return O.unpack_codes(qpacked.cpu().numpy().view(np.uint32), bits, d)


# ---------------------------------------------------------------------------------------
# Step 1: Hessian
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("d,n,dtype,dead,outl", [
    (256, 512, "f32", 0, 0),        # the 256 x 256, 512-token fp32 layer (3xTF32 tensor cores)
    (300, 777, "f32", 3, 2),        # fp32: ragged channels (a partial 128-wide tile) and tokens
    (1024, 4096, "f32", 10, 8),     # fp32: several segments of 512 tokens, 36 tiles
    (40, 100, "f32", 1, 1),         # fp32: one tile, mostly zero fill
    (300, 777, "f16", 3, 2),        # ragged channels and tokens
    (512, 2048, "bf16", 5, 4),
    (1024, 4096, "f16", 10, 8),
    (130, 64, "f16", 0, 0),
    # more 256 x 256 tiles than SM pairs: a partial last round
    (3200, 2048, "f16", 4, 3),      # 91 tiles; 4 segments: the last round is not cut
    (4096, 1000, "bf16", 0, 0),     # 136 tiles, 16 stages
    (4000, 640, "f16", 2, 1),       # ragged channels: the last rows of a pair beyond d
    (3998, 512, "f16", 0, 0),       # rows of H not 16-byte aligned
    # the last round's tiles cut into a head and a tail that add onto a zeroed H
    (4096, 4096, "f16", 0, 0),      # 60 cut tiles, heads of 6 of 8 segments, 4 tail batches
    (3000, 4100, "bf16", 3, 2),     # ragged channels and tokens: 2 cut tiles, tail ends ragged
])
def test_hessian_parity(d, n, dtype, dead, outl):
    spec = S.ActivationSpec(d_in=d, n_tok=n, dtype=dtype, n_dead=dead, n_outlier=outl, seed=d + n)
    X = _x(spec)
    if (d * X.element_size()) % 16:
        with pytest.raises(gptq.GptqError) as ei:   # unpadded row pitch is rejected
            gptq.hessian(X.to(DEV))
        assert ei.value.status == 1
    Hg = gptq.hessian(_padded(X))
    torch.cuda.synchronize()
    Hr = O.hessian(X.float().numpy() if dtype != "f32" else X.numpy())
    Hg = Hg.cpu().numpy()
    assert PT.rel_fro(Hg, Hr) <= PT.TOL_H
    assert np.array_equal(Hg, Hg.T)


def test_hessian_long_token_sum():
    # 262144 tokens into one H: the accumulation precision over a long sum
    spec = S.ActivationSpec(d_in=256, n_tok=262144, dtype="f16", n_dead=2, n_outlier=3, seed=91)
    Xg = S.activations(spec, device=DEV)
    Hg = gptq.hessian(Xg).cpu().numpy()
    Hr = O.hessian(Xg.cpu().float().numpy())
    assert PT.rel_fro(Hg, Hr) <= PT.TOL_H
    # diagonal entries (long sums of positive terms) individually
    dg, dr = np.diag(Hg), np.diag(Hr)
    live = dr > 0
    assert np.max(np.abs(dg[live] - dr[live]) / dr[live]) <= 1e-5


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_hessian_accumulates_over_chunks(dtype):
    spec = S.ActivationSpec(d_in=384, n_tok=6144, dtype=dtype, n_dead=2, seed=77)
    X = _x(spec).to(DEV)
    H = gptq.hessian(X[:2048])
    gptq.hessian(X[2048:4096], H, accumulate=True)
    gptq.hessian(X[4096:], H, accumulate=True)
    Hr = O.hessian(X.cpu().float().numpy())
    assert PT.rel_fro(H.cpu().numpy(), Hr) <= PT.TOL_H


def test_hessian_token_ranges_accumulate_over_chunks():
    # 91 tiles of 256 x 256: the first chunk's last round cut into heads and tails, the
    # later chunks (accumulating) uncut
    spec = S.ActivationSpec(d_in=3328, n_tok=6000, dtype="f16", n_dead=3, n_outlier=2, seed=78)
    X = _x(spec).to(DEV)
    H = gptq.hessian(X[:4096])
    gptq.hessian(X[4096:5000], H, accumulate=True)
    gptq.hessian(X[5000:], H, accumulate=True)
    Hr = O.hessian(X.cpu().float().numpy())
    Hg = H.cpu().numpy()
    assert PT.rel_fro(Hg, Hr) <= PT.TOL_H
    assert np.array_equal(Hg, Hg.T)


def test_hessian_cut_round_matches_uncut():
    # the same Hessian with the last round cut (overwrite) and uncut (accumulating onto
    # zeros): equal up to the grouping of the fp32 segment sums
    spec = S.ActivationSpec(d_in=4096, n_tok=4096, dtype="bf16", n_dead=2, n_outlier=2, seed=79)
    X = _x(spec).to(DEV)
    Hc = gptq.hessian(X)
    Hu = torch.zeros_like(Hc)
    gptq.hessian(X, Hu, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(Hc, Hc.T)
    assert ((Hc - Hu).abs().max() / Hu.abs().max()).item() <= 1e-6
    # a repeat of the cut call is bit-identical
    assert torch.equal(gptq.hessian(X), Hc)


def test_hessian_zero_tokens():
    H = torch.full((40, 40), 3.0, device=DEV)
    X = torch.empty(0, 40, dtype=torch.float16, device=DEV)
    gptq.hessian(X, H, accumulate=True)
    assert torch.all(H == 3.0)
    gptq.hessian(X, H, accumulate=False)
    assert torch.all(H == 0.0)


@pytest.mark.parametrize("d,n,dtype,chunk,ld_pad", [
    (384, 5000, "f16", 1024, 0),     # five chunks, ragged last one
    (256, 3000, "bf16", 512, 5),     # strided host rows
    (128, 700, "f32", 0, 0),         # default chunk: a single copy
    (1024, 4096, "f16", 1536, 0),    # chunks not a multiple of the drain segment
])
def test_hessian_host_streamed(d, n, dtype, chunk, ld_pad):
    spec = S.ActivationSpec(d_in=d, n_tok=n, dtype=dtype, n_dead=3, n_outlier=2, seed=d + n + 5)
    X = _x(spec)
    Xh = torch.zeros(n, d + ld_pad, dtype=X.dtype).pin_memory()
    Xh[:, :d] = X
    Hg = gptq.hessian_host(Xh[:, :d], chunk_tok=chunk, device=DEV)
    torch.cuda.synchronize()
    Hr = O.hessian(X.float().numpy() if dtype != "f32" else X.numpy())
    Hg = Hg.cpu().numpy()
    assert PT.rel_fro(Hg, Hr) <= PT.TOL_H
    assert np.array_equal(Hg, Hg.T)
    # one chunk holding every token is the device-resident call, bit for bit
    if chunk == 0:
        Hd = gptq.hessian(_padded(X)).cpu().numpy()
        assert np.array_equal(Hg, Hd)


def test_hessian_host_accumulates_and_reuses_workspace():
    spec = S.ActivationSpec(d_in=320, n_tok=4000, dtype="f16", n_dead=1, seed=33)
    X = _x(spec).pin_memory()
    ws = gptq.workspace(gptq.gptq_hessian_host_workspace_bytes(0, 320, 768), DEV)
    H = gptq.hessian_host(X[:1500], chunk_tok=768, ws=ws, device=DEV)
    gptq.hessian_host(X[1500:], H, accumulate=True, chunk_tok=768, ws=ws)
    Hr = O.hessian(X.float().numpy())
    assert PT.rel_fro(H.cpu().numpy(), Hr) <= PT.TOL_H
    # zero tokens: accumulate keeps H, otherwise H is cleared
    H2 = torch.full((320, 320), 3.0, device=DEV)
    gptq.hessian_host(X[:0], H2, accumulate=True, chunk_tok=768, ws=ws)
    assert torch.all(H2 == 3.0)
    gptq.hessian_host(X[:0], H2, accumulate=False, chunk_tok=768, ws=ws)
    assert torch.all(H2 == 0.0)


# ---------------------------------------------------------------------------------------
# Steps 2-3: dead columns, damping, U
# ---------------------------------------------------------------------------------------

def _oracle_h(d, n, dead, outl, seed, dtype="f16", relu=False):
    spec = S.ActivationSpec(d_in=d, n_tok=n, dtype=dtype, n_dead=dead, n_outlier=outl,
                            relu_t4=relu, seed=seed)
    X = _x(spec).float().numpy()
    return O.hessian(X)


@pytest.mark.parametrize("d,n,dead,outl", [
    (256, 512, 0, 0), (300, 900, 3, 2), (777, 3000, 7, 4), (1024, 4096, 10, 8),
    # wide enough for deferred groups: the columns past the next group of four panels are
    # updated once per group by the far products (one group, ragged; then three groups)
    (1600, 4096, 6, 3), (2560, 4096, 0, 2)])
def test_prepare_parity(d, n, dead, outl):
    H64 = _oracle_h(d, n, dead, outl, seed=d)
    H32 = H64.astype(np.float32)
    Hd, dmask, lam = O.damp_hessian(H32.astype(np.float64))
    Ur = O.inverse_cholesky_upper(Hd)
    Hg = torch.from_numpy(H32).to(DEV)
    U, mask, n_dead = gptq.prepare(Hg, 0.01)
    U = U.cpu().numpy()
    assert n_dead == dead
    assert np.array_equal(mask.cpu().numpy().astype(bool), dmask)
    assert np.all(np.tril(U, -1) == 0)
    assert PT.u_rowwise_err(U, Ur) <= PT.TOL_U


def test_prepare_relu_t4_inputs():
    H64 = _oracle_h(640, 4096, 0, 0, seed=5, relu=True)
    H32 = H64.astype(np.float32)
    Ur = O.inverse_cholesky_upper(O.damp_hessian(H32.astype(np.float64))[0])
    U, _, _ = gptq.prepare(torch.from_numpy(H32).to(DEV), 0.01)
    assert PT.u_rowwise_err(U.cpu().numpy(), Ur) <= PT.TOL_U


def test_prepare_not_positive_definite():
    H = torch.eye(200, device=DEV)
    H[150, 150] = -50.0
    with pytest.raises(gptq.GptqError) as ei:
        gptq.prepare(H, 0.0)
    assert ei.value.status == 2


def test_prepare_nonfinite():
    H = torch.eye(64, device=DEV)
    H[3, 5] = float("nan")
    with pytest.raises(gptq.GptqError) as ei:
        gptq.prepare(H, 0.01)
    assert ei.value.status == 3


def test_prepare_nonfinite_diagonal():
    H = torch.eye(65, device=DEV)
    H[64, 64] = float("inf")
    with pytest.raises(gptq.GptqError) as ei:
        gptq.prepare(H, 0.01)
    assert ei.value.status == 3


@pytest.mark.parametrize("d", [301, 512])     # odd (scalar path), and the float4 path
def test_prepare_reads_only_the_upper_triangle(d):
    # NaN below the diagonal changes nothing; the dead column sits at the middle of the
    # order reversal (for odd d the entry that maps to itself)
    H64 = _oracle_h(d, 2 * d, 2, 1, seed=40 + d)
    mid = d // 2
    H64[mid, :] = 0.0
    H64[:, mid] = 0.0
    H32 = H64.astype(np.float32)
    Hd, dmask, _ = O.damp_hessian(H32.astype(np.float64))
    Ur = O.inverse_cholesky_upper(Hd)
    Hn = H32.copy()
    Hn[np.tril_indices(d, -1)] = np.nan
    U, mask, n_dead = gptq.prepare(torch.from_numpy(Hn).to(DEV), 0.01)
    mask = mask.cpu().numpy().astype(bool)
    assert mask[mid] and np.array_equal(mask, dmask) and n_dead == int(dmask.sum())
    U = U.cpu().numpy()
    assert np.all(np.tril(U, -1) == 0)
    assert PT.u_rowwise_err(U, Ur) <= PT.TOL_U


# ---------------------------------------------------------------------------------------
# Steps 4-5 (+ packing): the sweep, on the oracle's U
# ---------------------------------------------------------------------------------------

def _quant_case(m, d, bits, block, wdtype, seed, dead=0, outl=0, n=None):
    H64 = _oracle_h(d, n or 2 * d, dead, outl, seed=seed)
    Hd, dmask, _ = O.damp_hessian(H64)
    U32 = O.inverse_cholesky_upper(Hd).astype(np.float32)
    W = S.weights(m, d, 0.02, wdtype, seed)
    return W, U32, dmask


@pytest.mark.parametrize("m,d,bits,block,wdtype", [
    (256, 256, 4, 128, "f32"),
    (200, 300, 4, 128, "bf16"),
    (64, 257, 3, 128, "bf16"),
    (130, 384, 2, 128, "f16"),
    (96, 200, 8, 128, "bf16"),
    (100, 256, 4, 32, "bf16"),
    (70, 150, 3, 7, "f32"),
    (33, 65, 4, 1, "f32"),
])
def test_quantize_parity(m, d, bits, block, wdtype):
    W, U32, dmask = _quant_case(m, d, bits, block, wdtype, seed=m * 7 + d, dead=2, outl=1)
    dm = torch.from_numpy(dmask.astype(np.uint8)).to(DEV)
    qp, sc, zr, Wh = gptq.quantize(W.to(DEV), torch.from_numpy(U32).to(DEV), bits, block, dm)
    torch.cuda.synchronize()
    Wn = W.float().numpy()
    s_ref, z_ref = O.row_grid(Wn, bits)
    assert np.array_equal(sc.cpu().numpy(), s_ref)          # grid is bit-exact
    assert np.array_equal(zr.cpu().numpy(), z_ref)
    codes = _codes(qp, bits, d)
    # packing layout: the oracle's packing of these codes gives the same words
    assert np.array_equal(O.pack_codes(codes, bits), qp.cpu().numpy().view(np.uint32))
    st = PT.check_codes(codes, Wn, U32.astype(np.float64), s_ref, z_ref, bits, block, dmask)
    # W_hat is the dequantized code, in fp32
    Wh_ref = (s_ref[:, None] * (codes - z_ref[:, None]).astype(np.float32)).astype(np.float32)
    assert np.array_equal(Wh.cpu().numpy(), Wh_ref)
    assert st["entries"] == m * d


def test_quantize_dead_columns_quantize_to_zero():
    W, U32, dmask = _quant_case(64, 256, 4, 128, "bf16", seed=3, dead=6)
    dm = torch.from_numpy(dmask.astype(np.uint8)).to(DEV)
    qp, sc, zr, Wh = gptq.quantize(W.to(DEV), torch.from_numpy(U32).to(DEV), 4, 128, dm)
    Wh = Wh.cpu().numpy()
    assert np.all(Wh[:, dmask] == 0.0)


def test_quantize_nonfinite_weights_flagged():
    W = torch.zeros(8, 64, device=DEV)
    W[2, 7] = float("inf")
    U = torch.eye(64, device=DEV)
    ws = gptq.workspace(gptq.gptq_quantize_workspace_bytes(8, 64, 4, 128), DEV)
    gptq.quantize(W, U, 4, 128, ws=ws)
    st = gptq.gptq_workspace_status(gptq._ptr(ws), gptq._stream(None))
    assert st == 3


# ---------------------------------------------------------------------------------------
# The whole path on the 256 x 256, 512-token layer
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [3, 4])
def test_layer_end_to_end_small(bits):
    wl = S.WORKLOADS["layer256_n512"]
    layer = wl.layers[0]
    X = S.activations(layer.act, device="cpu")
    W = S.layer_weights(layer)
    ref = O.gptq_layer(X.numpy(), W.numpy(), bits)
    Xg, Wg = X.to(DEV), W.to(DEV)
    H = gptq.hessian(Xg)
    U, dm, nd = gptq.prepare(H, 0.01)
    qp, sc, zr, Wh = gptq.quantize(Wg, U, bits, 128, dm)
    torch.cuda.synchronize()
    e_gpu = O.reconstruction_error(W.numpy(), Wh.cpu().numpy(), ref["H"])
    e_ref = O.reconstruction_error(W.numpy(), ref["W_hat"], ref["H"])
    assert abs(e_gpu - e_ref) <= PT.TOL_RECON * e_ref
    _, q_rtn = O.rtn_quantize(W.numpy(), ref["scale"], ref["zero"], bits)
    assert e_gpu < O.reconstruction_error(W.numpy(), q_rtn, ref["H"])
    assert nd == 0


# ---------------------------------------------------------------------------------------
# Layers sharing one Hessian: the shared sweep and the block driver
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("block", [128, 32, 1])
def test_quantize_shared_equals_separate_calls(block):
    d = 384
    _, U32, dmask = _quant_case(8, d, 4, block, "f32", seed=17, dead=3, outl=1)
    U = torch.from_numpy(U32).to(DEV)
    dm = torch.from_numpy(dmask.astype(np.uint8)).to(DEV)
    Ws = [S.weights(96, d, 0.02, "bf16", 1).to(DEV), S.weights(130, d, 0.02, "f16", 2).to(DEV),
          _padded(S.weights(64, d, 0.02, "f32", 3)), S.weights(1, d, 0.02, "bf16", 4).to(DEV)]
    for bits in (3, 4):
        shared = gptq.quantize_shared(Ws, U, bits, block, dm, want_w_hat=True)
        sep = [gptq.quantize(W, U, bits, block, dm) for W in Ws]
        torch.cuda.synchronize()
        for a, b in zip(shared, sep):
            for x, y in zip(a, b):
                assert torch.equal(x, y)


def test_quantize_block_driver_matches_per_layer_path():
    # two input streams: a 3-layer group and a 2-layer group, 3- and 4-bit
    specs = [S.ActivationSpec(d_in=256, n_tok=3000, dtype="f16", n_dead=2, n_outlier=1, seed=41),
             S.ActivationSpec(d_in=320, n_tok=2500, dtype="f16", n_dead=1, n_outlier=2, seed=42)]
    groups = []
    for i, sp in enumerate(specs):
        X = S.activations(sp, device=DEV)
        Ws = [S.weights(64 + 16 * j, sp.d_in, 0.02, "bf16", 10 * i + j).to(DEV)
              for j in range(3 - i)]
        groups.append((X, Ws))
    for overlap in (True, False):
        res, nd = gptq.quantize_block(groups, bits=(3, 4), overlap=overlap)
        torch.cuda.synchronize()
        for (X, Ws), r, n_dead in zip(groups, res, nd):
            U, dm, nd_ref = gptq.prepare(gptq.hessian(X), 0.01)
            assert n_dead == nd_ref
            for bits in (3, 4):
                for W, got in zip(Ws, r[bits]):
                    ref = gptq.quantize(W, U, bits, 128, dm, want_w_hat=False)
                    for x, y in zip(got[:3], ref[:3]):
                        assert torch.equal(x, y)


# ---------------------------------------------------------------------------------------
# The consumer: per-row ||(W - W_hat) X^T||^2 from the packed codes, on X
# ---------------------------------------------------------------------------------------

# W - W_hat is rounded to the activations' type before the tensor-core product (relative
# error <= u = 2^-11 fp16, 2^-8 bf16 per entry).  With delta' = delta (1 + eps) the row
# error moves by 2 delta H (delta o eps) + O(u^2), at most 2u of it: tolerance 2.5 u.
REL_TOL = {"f16": 2.5 * 2.0 ** -11, "bf16": 2.5 * 2.0 ** -8, "f32": 1e-5}


@pytest.mark.parametrize("m,d,n,bits,xdtype", [
    (96, 384, 1000, 4, "f16"),
    (130, 200, 777, 3, "f16"),      # ragged rows, tokens and K
    (64, 256, 700, 3, "bf16"),
    (256, 256, 512, 4, "f32"),      # the 256 x 256 fp32 layer
    (300, 512, 3000, 2, "f16"),
])
def test_recon_error_parity(m, d, n, bits, xdtype):
    spec = S.ActivationSpec(d_in=d, n_tok=n, dtype=xdtype, n_dead=2, n_outlier=1, seed=m + d)
    X = _x(spec)
    Xn = X.float().numpy() if xdtype != "f32" else X.numpy()
    W = S.weights(m, d, 0.02, "bf16", m + n)
    U, dm, _ = gptq.prepare(gptq.hessian(_padded(X)), 0.01)
    Wg = W.to(DEV)
    qp, sc, zr, Wh = gptq.quantize(Wg, U, bits, 128, dm)
    err = gptq.recon_error(_padded(X), Wg, qp, bits, sc, zr)
    err2 = gptq.recon_error(_padded(X), Wg, qp, bits, sc, zr)
    torch.cuda.synchronize()
    ref = O.reconstruction_error_rows(W.float().numpy(), Wh.cpu().numpy(), Xn)
    got = err.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref) / np.maximum(ref, 1e-30)) <= REL_TOL[xdtype]
    assert torch.equal(err, err2)     # fixed-order reduction: repeatable


def test_recon_error_zero_tokens():
    d, m = 256, 64
    X = torch.empty(0, d, dtype=torch.float16, device=DEV)
    W = S.weights(m, d, 0.02, "bf16", 3).to(DEV)
    U = torch.eye(d, device=DEV)
    qp, sc, zr, _ = gptq.quantize(W, U, 4, 128)
    assert torch.all(gptq.recon_error(X, W, qp, 4, sc, zr) == 0)


# ---------------------------------------------------------------------------------------
# OBQ greedy order: the GPU's order and codes replayed through the oracle
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("m,d,bits,wdtype,dead", [
    (64, 64, 4, "bf16", 2),
    (100, 128, 3, "f32", 3),
    (33, 37, 2, "f16", 1),          # ragged width
    (40, 1, 4, "f32", 0),           # a single column
])
def test_obq_parity(m, d, bits, wdtype, dead):
    W, U32, dmask = _quant_case(m, d, bits, 128, wdtype, seed=m + 3 * d, dead=dead, outl=1)
    Hd = np.linalg.inv(U32.astype(np.float64).T @ U32.astype(np.float64))
    dm = torch.from_numpy(dmask.astype(np.uint8)).to(DEV)
    Wg = W.to(DEV) if (d * W.element_size()) % 16 == 0 else _padded(W)
    qp, sc, zr, Wh, order = gptq.quantize_obq(Wg, torch.from_numpy(U32).to(DEV), bits, dm)
    torch.cuda.synchronize()
    Wn = W.float().numpy()
    s_ref, z_ref = O.row_grid(Wn, bits)
    assert np.array_equal(sc.cpu().numpy(), s_ref)
    assert np.array_equal(zr.cpu().numpy(), z_ref)
    codes = _codes(qp, bits, d)
    order = order.cpu().numpy().astype(np.int64)
    for i in range(m):
        assert sorted(order[i]) == list(range(d))
    _, _, _, info = O.obq_greedy(Wn, Hd, s_ref, z_ref, bits, dead=dmask, forced=(order, codes))
    assert info["bad_order"] == 0 and info["bad_codes"] == 0
    assert info["max_slack"] <= 1e-4
    assert info["tie_flips"] <= max(1, m * d // 5000)
    Wh_ref = (s_ref[:, None] * (codes - z_ref[:, None]).astype(np.float32)).astype(np.float32)
    assert np.array_equal(Wh.cpu().numpy(), Wh_ref)
