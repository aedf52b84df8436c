"""Failure paths on the GPU that fault, trap and hang nothing.

Every wait inside the tensor-core kernels is bounded in time.  The library's test hook
gptq_debug_hessian_lost_stage runs the Hessian kernel with its copy producer skipping one
token stage, so that the MMA issuer's wait for that stage can never complete; with a short
budget every wait then gives up, the kernel records GPTQ_ERR_TIMEOUT and returns, and the
context stays usable: the next regular call on the same GPU gives the exact Hessian.
"""

import ctypes
import time

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


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("d,n,lost", [(256, 4096, 10), (384, 1000, 5), (128, 640, 0)])
def test_lost_stage_times_out_and_context_survives(d, n, lost):
    spec = S.ActivationSpec(d_in=d, n_tok=n, dtype="f16", n_dead=1, n_outlier=1, seed=d + n)
    X = S.activations(spec, device=DEV)
    H = torch.empty(d, d, dtype=torch.float32, device=DEV)
    status = gptq.workspace(256, DEV)
    t0 = time.time()
    st = gptq.gptq_debug_hessian_lost_stage(_p(X), 0, n, d, X.stride(0), _p(H), lost,
                                            50_000_000, _p(status), gptq._stream(None))
    elapsed = time.time() - t0
    assert st == 4, gptq.gptq_status_str(st)      # GPTQ_ERR_TIMEOUT
    assert elapsed < 5.0                            # a few 50 ms budgets, not the 2 s default
    # the same GPU, next regular call: the exact Hessian
    Hg = gptq.hessian(X)
    torch.cuda.synchronize()
    assert PT.rel_fro(Hg.cpu().numpy(), O.hessian(X.cpu().float().numpy())) <= PT.TOL_H


def test_lost_stage_hook_rejects_bad_requests():
    X = torch.zeros(128, 64, dtype=torch.float16, device=DEV)
    H = torch.empty(64, 64, dtype=torch.float32, device=DEV)
    status = gptq.workspace(256, DEV)
    s = gptq._stream(None)
    # fp32 inputs do not take the fp16/bf16 tensor-core kernel
    Xf = torch.zeros(128, 64, dtype=torch.float32, device=DEV)
    assert gptq.gptq_debug_hessian_lost_stage(_p(Xf), 2, 128, 64, 64, _p(H), 0, 10**6,
                                              _p(status), s) == 6
    # stage out of range, budget out of range
    assert gptq.gptq_debug_hessian_lost_stage(_p(X), 0, 128, 64, 64, _p(H), 2, 10**6,
                                              _p(status), s) == 1
    assert gptq.gptq_debug_hessian_lost_stage(_p(X), 0, 128, 64, 64, _p(H), 0, 10,
                                              _p(status), s) == 1
    # nothing was launched: a regular call still works
    assert torch.all(gptq.hessian(X) == 0)
