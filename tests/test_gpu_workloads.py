"""GPU parity at the full sizes of the five layer workloads.

Where the fp64 oracle cannot redo the whole computation at full size, the check is one the
oracle can afford:
  * Hessian: exact sub-Gram blocks of sampled channels (dead, outlier and random ones) and
    the exact diagonal, from the same fp16 activation bits;
  * factor: U's trailing k x k block depends only on the trailing block of the damped H
    (pinned in the oracle tests), so it is checked against the oracle's factor of that
    block, damped with lambda from the full exact diagonal;
  * sweep: the oracle's U (at d_in = 4096, from a token prefix) or a seeded synthetic upper
    factor (d_in = 11008, 28672) as the shared input, the oracle sweeping sampled rows (at
    d_in = 4096 also with B = 1, the eager column-at-a-time variant);
  * the consumer (per-row output error from the packed codes) over all tokens, sampled rows
    against the oracle;
  * shared-Hessian batching: rows of q/k/v (and gate/up) quantized in one call (stacked
    rows, or the shared multi-layer call) equal the separate calls bit for bit (rows
    decouple: "GPTQ Hessian").
"""

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as O
from post_weight_quantization_03_gb300 import build_lib, gptq
from post_weight_quantization_03_gb300 import synthetic as S
from tests import parity as PT

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda:0"
TAIL = 512


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    gptq.load()
    torch.cuda.init()


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _sample_channels(act, n_random=88, seed=0):
    dead, outl = S.channel_roles(act)
    rng = np.random.default_rng(seed)
    ch = np.concatenate([dead.numpy()[:3], outl.numpy()[:5],
                         rng.choice(act.d_in, n_random, replace=False),
                         np.arange(act.d_in - 8, act.d_in)])
    return np.unique(ch)


def _check_hessian(Xg, Hg, act):
    ch = _sample_channels(act)
    Xs = Xg[:, torch.from_numpy(ch).to(DEV)].cpu().numpy()
    ref = O.hessian_block(Xs, slice(None), slice(None))
    got = Hg[torch.from_numpy(ch).to(DEV)][:, torch.from_numpy(ch).to(DEV)].cpu().numpy()
    assert PT.rel_fro(got, ref) <= PT.TOL_H
    assert np.array_equal(got, got.T)


def _check_factor_tail(Xh, diag_full, U, dmask, n_dead, damp=0.01):
    d = Xh.shape[1]
    tail = np.arange(d - TAIL, d)
    Hb = O.hessian_block(Xh, tail, tail)
    Hbd, dead, _ = O.damp_principal_block(Hb, diag_full, tail, damp)
    Ut = O.inverse_cholesky_upper(Hbd)
    got = U[d - TAIL:, d - TAIL:].cpu().numpy()
    assert PT.u_rowwise_err(got, Ut) <= PT.TOL_U
    assert np.array_equal(dmask.cpu().numpy().astype(bool), dead)
    assert n_dead == int(dead.sum())
    Uh_diag = torch.diagonal(U).cpu().numpy()
    assert np.all(Uh_diag > 0)


def _quantize_and_check(W, U32_np, dead, bits, rows, block=128):
    Ug = torch.from_numpy(U32_np).to(DEV)
    dm = torch.from_numpy(dead.astype(np.uint8)).to(DEV) if dead is not None else None
    qp, sc, zr, _ = gptq.quantize(W, Ug, bits, block, dm, want_w_hat=False)
    torch.cuda.synchronize()
    Wn = W.float().cpu().numpy()
    s_ref, z_ref = O.row_grid(Wn[rows], bits)
    assert np.array_equal(sc.cpu().numpy()[rows], s_ref)
    assert np.array_equal(zr.cpu().numpy()[rows], z_ref)
    codes = O.unpack_codes(qp[torch.from_numpy(rows).to(DEV)].cpu().numpy().view(np.uint32), bits,
                           W.shape[1])
    st = PT.check_codes(codes, Wn[rows], U32_np.astype(np.float64), s_ref, z_ref, bits, block,
                        dead)
    return st


# ---------------------------------------------------------------------------------------

def test_layer4096_n262144():
    wl = S.WORKLOADS["layer4096_n262144"]
    layer, bits = wl.layers[0], wl.bits[0]
    act = layer.act
    Xg = S.activations(act, device=DEV)
    Hg = gptq.hessian(Xg)
    _check_hessian(Xg, Hg, act)
    Xh = Xg.cpu().numpy()
    diag_full = O.hessian_diagonal(Xh)
    # factor of the full-size GPU Hessian, trailing block against the oracle
    U, dm, nd = gptq.prepare(Hg, wl.damp)
    assert nd == act.n_dead
    _check_factor_tail(Xh, diag_full, U, dm, nd)
    del U, Hg
    _free()
    # sweep of all 4096 rows on the oracle's U (from a 16384-token prefix)
    Xp = Xh[:16384]
    Hp = O.hessian(Xp)
    Hpd, dead_p, _ = O.damp_hessian(Hp, wl.damp)
    U32 = O.inverse_cholesky_upper(Hpd).astype(np.float32)
    W = S.layer_weights(layer, DEV)
    st = _quantize_and_check(W, U32, dead_p, bits, np.arange(layer.d_out))
    assert st["entries"] == 4096 * 4096
    # the eager variant (B = 1: a rank-1 update of every later column after each column),
    # sampled rows against the oracle's column-at-a-time sweep
    rows = np.sort(np.random.default_rng(5).choice(layer.d_out, 48, replace=False))
    _quantize_and_check(W, U32, dead_p, bits, rows, block=1)
    # the whole path on the prefix: reconstruction error within 0.1 % of the oracle's
    Hg = gptq.hessian(Xg[:16384])
    U, dm, _ = gptq.prepare(Hg, wl.damp)
    qp, sc, zr, Wh = gptq.quantize(W, U, bits, 128, dm)
    Wn = W.float().cpu().numpy()
    ref = O.gptq_quantize(Wn, O.inverse_cholesky_upper(Hpd), *O.row_grid(Wn, bits), bits,
                          block=128, dead=dead_p)[1]
    e_gpu = O.reconstruction_error(Wn, Wh.cpu().numpy(), Hp)
    e_ref = O.reconstruction_error(Wn, ref, Hp)
    assert abs(e_gpu - e_ref) <= PT.TOL_RECON * e_ref
    # the consumer on all 262144 tokens, sampled rows against the oracle (token chunks)
    err = gptq.recon_error(Xg, W, qp, bits, sc, zr).cpu().numpy().astype(np.float64)
    rows = np.sort(np.random.default_rng(6).choice(layer.d_out, 24, replace=False))
    chunks = [Xh[t:t + 32768] for t in range(0, Xh.shape[0], 32768)]
    ref_rows = O.reconstruction_error_rows(Wn[rows], Wh.cpu().numpy()[rows], chunks)
    assert np.max(np.abs(err[rows] - ref_rows) / ref_rows) <= 2.5 * 2.0 ** -11


def test_mlp11008_n131072():
    wl = S.WORKLOADS["mlp11008_n131072"]
    up, down = wl.layers
    bits = wl.bits[0]
    # up-proj (11008 x 4096): oracle U from an 8192-token prefix of its inputs
    Xu = S.activations(up.act, device="cpu", n_tok=8192).numpy()
    Hd, dead, _ = O.damp_hessian(O.hessian(Xu), wl.damp)
    U32 = O.inverse_cholesky_upper(Hd).astype(np.float32)
    W = S.layer_weights(up, DEV)
    rows = np.random.default_rng(1).choice(up.d_out, 384, replace=False)
    _quantize_and_check(W, U32, dead, bits, np.sort(rows))
    del W
    _free()
    # down-proj (4096 x 11008, ReLU-sparse Student-t inputs): full-size Hessian + factor
    Xg = S.activations(down.act, device=DEV)
    Hg = gptq.hessian(Xg)
    _check_hessian(Xg, Hg, down.act)
    Xh = Xg.cpu().numpy()
    del Xg
    diag_full = O.hessian_diagonal(Xh)
    U, dm, nd = gptq.prepare(Hg, wl.damp)
    _check_factor_tail(Xh, diag_full, U, dm, nd)
    del U, Hg, Xh
    _free()
    # sweep at d_in = 11008 on a synthetic factor, sampled rows
    Us = S.upper_factor(down.act.d_in, 11, device="cpu").numpy()
    W = S.layer_weights(down, DEV)
    rows = np.sort(np.random.default_rng(2).choice(down.d_out, 48, replace=False))
    _quantize_and_check(W, Us, None, bits, rows)


def test_block7b_n131072():
    wl = S.WORKLOADS["block7b_n131072"]
    by_name = {l.name: l for l in wl.layers}
    # one Hessian per input stream; sampled exact checks
    for name in ("q_proj", "o_proj", "gate_proj", "down_proj"):
        act = by_name[name].act
        Xg = S.activations(act, device=DEV)
        Hg = gptq.hessian(Xg)
        _check_hessian(Xg, Hg, act)
        del Xg, Hg
        _free()
    # shared-H batching (q/k/v, gate/up): one call on concatenated rows == separate calls
    for group in (("q_proj", "k_proj", "v_proj"), ("gate_proj", "up_proj")):
        act = by_name[group[0]].act
        Xg = S.activations(act, device=DEV)
        U, dm, _ = gptq.prepare(gptq.hessian(Xg), wl.damp)
        del Xg
        Ws = [S.layer_weights(by_name[n], DEV) for n in group]
        for bits in wl.bits:
            sep = [gptq.quantize(w, U, bits, 128, dm, want_w_hat=False) for w in Ws]
            cat = gptq.quantize(torch.cat(Ws), U, bits, 128, dm, want_w_hat=False)
            shared = gptq.quantize_shared(Ws, U, bits, 128, dm)
            torch.cuda.synchronize()
            for k in range(3):
                assert torch.equal(cat[k], torch.cat([s[k] for s in sep]))
                assert torch.equal(cat[k], torch.cat([s[k] for s in shared]))
        del U, Ws
        _free()
    # o_proj at 3 and 4 bits against the oracle (U from an 8192-token prefix), sampled rows
    o = by_name["o_proj"]
    Xo = S.activations(o.act, device="cpu", n_tok=8192).numpy()
    Hd, dead, _ = O.damp_hessian(O.hessian(Xo), wl.damp)
    U32 = O.inverse_cholesky_upper(Hd).astype(np.float32)
    W = S.layer_weights(o, DEV)
    rows = np.sort(np.random.default_rng(3).choice(o.d_out, 256, replace=False))
    for bits in wl.bits:
        _quantize_and_check(W, U32, dead, bits, rows)


def test_downproj28672_n65536():
    wl = S.WORKLOADS["downproj28672_n65536"]
    layer, bits = wl.layers[0], wl.bits[0]
    act = layer.act
    Xg = S.activations(act, device=DEV)
    Hg = gptq.hessian(Xg)
    _check_hessian(Xg, Hg, act)
    Xh = Xg.cpu().numpy()
    del Xg
    _free()
    diag_full = O.hessian_diagonal(Xh)
    U, dm, nd = gptq.prepare(Hg, wl.damp)
    assert nd == act.n_dead
    _check_factor_tail(Xh, diag_full, U, dm, nd)
    del U, Hg, Xh
    _free()
    Us = S.upper_factor(act.d_in, 28, device="cpu").numpy()
    W = S.layer_weights(layer, DEV)
    rows = np.sort(np.random.default_rng(4).choice(layer.d_out, 12, replace=False))
    _quantize_and_check(W, Us, None, bits, rows)
