"""e4m3 (fp8) forward: the row quantiser bit for bit against the oracle's
definition, and the e4m3 forward against the oracle on the same quantised
operands."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import LOSS_RTOL, assert_logp_close, np64, run_forward, to_dev_bf16, upload

pytestmark = pytest.mark.gpu


def _quantize_dev(x_dev):
    rows, cols = x_dev.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    assert _lib.flce_quantize_e4m3_rows(x_dev, rows, cols, q, s) == 0
    assert _lib.flce_device_status() == 0
    return q, s


def test_quantiser_is_bit_exact():
    r = np.random.default_rng(9)
    x = (r.standard_normal((300, 272)) * np.exp(2 * r.standard_normal((300, 1)))).astype(np.float32)
    x[5] = 0.0
    x[6, :3] = [1e30, -1e30, 3.0]
    bits = WL.f32_to_bf16_bits(x)
    q, s = _quantize_dev(to_dev_bf16(bits))
    q_ref, s_ref = O.quantize_e4m3_rows(bits)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("cg", ["1", "2"])
@pytest.mark.parametrize("shape,tfd", [((300, 192, 2100), None), ((520, 512, 3000), {"softcap": 20.0})])
def test_e4m3_forward_parity(cg, shape, tfd, flce_opts):
    flce_opts.set("cta_group", cg)
    N, H, V = shape
    wl = WL.custom("e4m3", N, H, V, 256, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=700 + N)
    inp = WL.make_inputs(wl)
    h, W, t, _ = upload(inp)
    h8, hs = _quantize_dev(h)
    W8, Ws = _quantize_dev(W)
    logp = torch.empty(N, dtype=torch.float32, device="cuda")
    lse = torch.empty(N, dtype=torch.float32, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    nv = torch.empty(1, dtype=torch.int64, device="cuda")
    st = _lib.flce_forward_e4m3(h8, hs, W8, Ws, t, None, N, H, V, 256, -100, tfd, logp, lse, loss, nv)
    assert st == 0 and _lib.flce_device_status() == 0
    tf = None if tfd is None else O.LogitTransform(**tfd)
    ref = O.forward_fp8(h8.cpu().numpy(), hs.cpu().numpy(), W8.cpu().numpy(), Ws.cpu().numpy(),
                        inp.targets, tf=tf)
    assert int(nv.item()) == ref.n_valid
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert_logp_close(np64(lse), ref.lse, "lse")
    assert float(loss.item()) == pytest.approx(ref.loss, rel=LOSS_RTOL)
    # informational: e4m3 operands against the bf16 path on the same inputs
    logp16, _, _, _ = run_forward(h, W, t, None, 256, transform=tfd)
    drift = np.abs(np64(logp) - np64(logp16))
    assert np.mean(drift) < 0.05, np.mean(drift)
