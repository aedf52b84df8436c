"""The C-ABI library builds, loads and exports every symbol include/gptq.h declares.

No compute call runs here: only calls whose arguments fail validation, which the
library rejects synchronously before touching the GPU.
"""

import ctypes

import pytest

from post_weight_quantization_03_gb300 import build_lib, gptq


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return gptq.load()


def test_exports_every_declared_symbol(lib):
    names = gptq.declared_symbols()
    assert {"gptq_hessian_accumulate", "gptq_prepare", "gptq_quantize_layer"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in gptq._SIGS, f"binding lacks a signature for {n}"


def test_status_strings_and_version(lib):
    for code, name in gptq.STATUS_NAMES.items():
        assert gptq.gptq_status_str(code) == name
    assert gptq.gptq_status_str(99) == "GPTQ_ERR_UNKNOWN"
    assert gptq.gptq_abi_version() == 1
    assert gptq.gptq_kernel_launches() >= 0


def test_workspace_sizes(lib):
    assert gptq.gptq_prepare_workspace_bytes(0) == 0
    assert gptq.gptq_prepare_workspace_bytes(4096) >= 4096 * 4096 * 4
    q = gptq.gptq_quantize_workspace_bytes(4096, 4096, 4, 128)
    assert q >= 4096 * 4096 * 4 * 3  # fp32 working copy + split U^T
    assert gptq.gptq_quantize_workspace_bytes(0, 10, 4, 128) == 0
    # host-streamed Hessian: two staging buffers of chunk_tok rows (default ~64 MiB each,
    # a multiple of 512 tokens), 256-byte rounded
    assert gptq.gptq_hessian_host_workspace_bytes(0, 4096, 0) == 2 * 8192 * 4096 * 2
    assert gptq.gptq_hessian_host_workspace_bytes(0, 300, 1000) == 2 * 600064
    assert gptq.gptq_hessian_host_workspace_bytes(9, 4096, 0) == 0
    assert gptq.gptq_hessian_host_workspace_bytes(0, 0, 0) == 0
    assert gptq.gptq_hessian_host_workspace_bytes(0, 64, -1) == 0
    # shared sweep: the stacked rows' workspace plus the stacked scales and zeros
    rows = (ctypes.c_int64 * 3)(4096, 4096, 4096)
    assert gptq.gptq_quantize_shared_workspace_bytes(3, rows, 4096, 4, 128) == \
        gptq.gptq_quantize_workspace_bytes(12288, 4096, 4, 128) + 2 * 12288 * 4
    one = (ctypes.c_int64 * 1)(300)
    assert gptq.gptq_quantize_shared_workspace_bytes(1, one, 200, 3, 128) == \
        gptq.gptq_quantize_workspace_bytes(300, 200, 3, 128)
    assert gptq.gptq_quantize_shared_workspace_bytes(0, rows, 4096, 4, 128) == 0
    assert gptq.gptq_quantize_shared_workspace_bytes(65, rows, 4096, 4, 128) == 0


P = ctypes.c_void_p


def test_invalid_arguments_rejected_before_launch(lib):
    fake = P(256 * 1024)  # never dereferenced: validation fails first
    INV, WS = 1, 7
    # bad dtype, negative tokens, ldx < d_in, null H
    assert gptq.gptq_hessian_accumulate(fake, 9, 10, 8, 8, fake, 0, None) == INV
    assert gptq.gptq_hessian_accumulate(fake, 0, -1, 8, 8, fake, 0, None) == INV
    assert gptq.gptq_hessian_accumulate(fake, 0, 10, 8, 4, fake, 0, None) == INV
    assert gptq.gptq_hessian_accumulate(fake, 0, 10, 8, 8, None, 0, None) == INV
    # misaligned X row stride (f16, ldx = 9 -> 18 bytes)
    assert gptq.gptq_hessian_accumulate(fake, 0, 10, 8, 9, fake, 0, None) == INV
    # host-streamed Hessian: bad chunk size, d_in pitch not 16 bytes, workspace
    hh = gptq.gptq_hessian_accumulate_host
    assert hh(fake, 0, 10, 8, 8, fake, 0, -1, fake, 1 << 30, None) == INV
    assert hh(fake, 0, 10, 9, 9, fake, 0, 0, fake, 1 << 30, None) == INV
    assert hh(None, 0, 10, 8, 8, fake, 0, 0, fake, 1 << 30, None) == INV
    assert hh(fake, 0, 10, 8, 8, fake, 0, 64, fake, 16, None) == WS
    assert hh(fake, 0, 10, 8, 8, fake, 0, 64, P(256 * 1024 + 8), 1 << 30, None) == WS
    # shared multi-layer sweep: layer count, null arrays, bits, workspace
    import ctypes as C
    n1 = (C.c_int64 * 1)(4)
    arr = (C.c_void_p * 1)(256 * 1024)
    dts = (C.c_int * 1)(1)
    lds = (C.c_int64 * 1)(8)
    sh = gptq.gptq_quantize_layers_shared
    assert sh(0, arr, dts, n1, lds, 8, fake, None, 4, 128, arr, arr, arr, None, fake, 1 << 30,
              None) == INV
    assert sh(65, arr, dts, n1, lds, 8, fake, None, 4, 128, arr, arr, arr, None, fake, 1 << 30,
              None) == INV
    assert sh(1, None, dts, n1, lds, 8, fake, None, 4, 128, arr, arr, arr, None, fake, 1 << 30,
              None) == INV
    assert sh(1, arr, dts, n1, lds, 8, fake, None, 5, 128, arr, arr, arr, None, fake, 1 << 30,
              None) == INV
    assert sh(1, arr, dts, n1, (C.c_int64 * 1)(7), 8, fake, None, 4, 128, arr, arr, arr, None,
              fake, 1 << 30, None) == INV
    assert sh(1, arr, dts, n1, lds, 8, fake, None, 4, 128, arr, arr, arr, None, fake, 16,
              None) == WS
    # reconstruction error: dtype, bits, X pitch, workspace
    re = gptq.gptq_recon_error
    assert re(fake, 9, 10, 8, 8, fake, 1, 4, 8, fake, 4, fake, fake, fake, fake, 1 << 30,
              None) == INV
    assert re(fake, 0, 10, 8, 8, fake, 1, 4, 8, fake, 5, fake, fake, fake, fake, 1 << 30,
              None) == INV
    assert re(fake, 0, 10, 8, 9, fake, 1, 4, 8, fake, 4, fake, fake, fake, fake, 1 << 30,
              None) == INV
    assert re(fake, 0, 10, 8, 8, fake, 1, 4, 8, fake, 4, fake, fake, None, fake, 1 << 30,
              None) == INV
    assert re(fake, 0, 10, 8, 8, fake, 1, 4, 8, fake, 4, fake, fake, fake, fake, 16,
              None) == WS
    assert gptq.gptq_recon_error_workspace_bytes(0, 4096, 4096, 262144) >= \
        4096 * 4096 * 2 + 1024 * 4096 * 4
    assert gptq.gptq_recon_error_workspace_bytes(9, 4, 8, 10) == 0
    # OBQ: too wide, bits, workspace
    ob = gptq.gptq_quantize_obq
    assert ob(fake, 1, 4, 129, 129, fake, None, 4, fake, fake, fake, None, None, fake, 1 << 30,
              None) == 6
    assert ob(fake, 1, 4, 64, 64, fake, None, 6, fake, fake, fake, None, None, fake, 1 << 30,
              None) == INV
    assert ob(fake, 1, 4, 64, 64, fake, None, 4, fake, fake, fake, None, None, fake, 16,
              None) == WS
    assert gptq.gptq_quantize_obq_workspace_bytes(0, 64) == 0
    # prepare: negative damp, missing or short workspace
    assert gptq.gptq_prepare(fake, 8, -1.0, fake, None, None, fake, 1 << 20, None) == INV
    assert gptq.gptq_prepare(fake, 8, 0.01, fake, None, None, None, 0, None) == WS
    assert gptq.gptq_prepare(fake, 8, 0.01, fake, None, None, fake, 16, None) == WS
    assert gptq.gptq_prepare(fake, 8, 0.01, fake, None, None, P(256 * 1024 + 8), 1 << 30,
                             None) == WS
    # quantize: bits, block, shapes, workspace
    args = dict(W=fake, wdtype=1, d_out=4, d_in=8, ldw=8, U=fake, dead_mask=None, bits=4,
                block=128, qpacked=fake, scale=fake, zero=fake, W_hat=None, ws=fake,
                ws_bytes=1 << 30, stream=None)

    def q(**kw):
        a = dict(args)
        a.update(kw)
        return gptq.gptq_quantize_layer(*a.values())

    assert q(bits=5) == INV
    assert q(bits=1) == INV
    assert q(block=0) == INV
    assert q(block=129) == INV
    assert q(ldw=7) == INV
    assert q(d_out=0) == INV
    assert q(wdtype=7) == INV
    assert q(qpacked=None) == INV
    assert q(ws=None) == WS
    assert q(ws_bytes=10) == WS
