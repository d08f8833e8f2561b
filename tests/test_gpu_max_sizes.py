"""The operator and the activation quantiser at the header's size limits
(SVDQ_MAX_K = 2^20, SVDQ_MAX_MN = 2^24), through the C ABI: index arithmetic
(tile and row coordinates, byte offsets of operands, scales, LoRA rows and the
outputs) must not overflow.

The operator is separable: output rows depend only on their act / ascales /
lora_act_in rows, output columns only on their wgt / wscales / lora_up /
wcscale / bias entries.  So the oracle checks sampled rows (the first, the
last, every tile edge they span) or sampled columns by running on the
matching slice of the inputs.
"""

import numpy as np
import pytest
import torch

from gpu_util import oracle_y, parity, run_gpu
from nvfp4_w4a4_quantized_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import oracle
    from nvfp4_w4a4_quantized_gb300 import build
    build.build()
    oracle.build()


def _edges(n, extra, seed):
    rng = np.random.default_rng(seed)
    idx = {0, 1, 127, 128, 255, 256, n // 2, n - 129, n - 128, n - 2, n - 1}
    idx |= set(int(x) for x in rng.integers(0, n, extra))
    return sorted(i for i in idx if 0 <= i < n)


def test_max_k():
    M, N, K, R = 256, 256, binding.SVDQ_MAX_K, 16
    inp = synth.make_inputs(M, N, K, R, seed=21)
    y = run_gpu(inp, M, N, K, R)
    rows = _edges(M, 4, 1)
    parity(y[rows], oracle_y(inp, M, N, K, R, rows=rows))


def test_max_m():
    M, N, K, R = binding.SVDQ_MAX_MN, 16, 64, 8
    inp = synth.make_inputs(M, N, K, R, seed=22)
    y = run_gpu(inp, M, N, K, R)
    rows = _edges(M, 40, 2)
    parity(y[rows], oracle_y(inp, M, N, K, R, rows=rows))


def test_max_n():
    M, N, K, R = 16, binding.SVDQ_MAX_MN, 64, 8
    inp = synth.make_inputs(M, N, K, R, seed=23)
    y = run_gpu(inp, M, N, K, R)
    cols = _edges(N, 40, 3)
    sub = dict(inp, wgt=inp["wgt"][cols].contiguous(), wscales=inp["wscales"][:, cols].contiguous(),
               lora_up=inp["lora_up"][cols].contiguous(), wcscale=inp["wcscale"][cols].contiguous(),
               bias=inp["bias"][cols].contiguous())
    parity(y[:, cols], oracle_y(sub, M, len(cols), K, R))


def _quant_check(x, ld, M, K, R, rows):
    # the quantiser is separable by rows: codes, scales and LoRA-down of the
    # sampled rows against the oracle on those rows alone
    from oracle import quant_ref as q

    act, asc, la = binding.svdq_quantize_act(x.cuda(), ld.cuda() if R else None)
    torch.cuda.synchronize()
    code, site, _ = binding.svdq_read_device_status(clear=True)
    assert code == 0, (code, site)
    idx = torch.tensor(rows)
    xr = x[idx]
    want_act, want_asc = q.quantize_act(xr, len(rows), K)
    np.testing.assert_array_equal(act[idx.cuda()].cpu().numpy(), want_act)
    np.testing.assert_array_equal(asc[:, idx.cuda()].cpu().numpy(), want_asc)
    if R:
        ref = q.lora_down(xr, ld, len(rows), K, R)
        mag = np.abs(q.decode_x(xr, len(rows), K)) @ np.abs(q.decode_x(ld, R, K)).T
        err = np.abs(la[idx.cuda()].double().cpu().numpy() - ref)
        assert np.all(err <= K * 2.0 ** -22 * mag + 1e-30)


def test_quantiser_max_k():
    M, K, R = 16, binding.SVDQ_MAX_K, 32
    a = synth.make_activations(M, K, R, seed=24)
    _quant_check(a["x"], a["lora_down"], M, K, R, list(range(M)))


def test_quantiser_max_m():
    M, K, R = binding.SVDQ_MAX_MN, 64, 8
    a = synth.make_activations(M, K, R, seed=25)
    _quant_check(a["x"], a["lora_down"], M, K, R, _edges(M, 40, 4))
