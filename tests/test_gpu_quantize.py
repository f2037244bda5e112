"""RTN quantiser kernel against the oracle (bit-exact codes, scales and
zeros), and the static SVD initialisation run through the decode kernel."""
import numpy as np
import pytest
import torch

from oracle import ref, rtn
from quantized_linear_error_gb300 import calibrate, spear
from quantized_linear_error_gb300 import workload as wl

from .helpers import dev_bf16, host_f64, rel_err

pytestmark = pytest.mark.gpu


def _weights(seed, N, K):
    rng = np.random.default_rng(seed)
    w = rng.normal(0, 0.02, size=(N, K)).astype(np.float32)
    w[0] = 0.0                                         # all-zero row
    w[1] = 0.125                                       # constant positive row
    w[2] = np.linspace(0.25, 1.5, K, dtype=np.float32)  # positive ramp (range must include 0)
    w[3, ::7] *= 50.0                                  # outliers
    w[4] = -np.abs(w[4])                               # non-positive row
    return w


@pytest.mark.parametrize("group_size", [128, 0])
@pytest.mark.parametrize("N,K", [(8, 128), (40, 384), (130, 2048)])
def test_rtn_bit_exact(N, K, group_size):
    w = _weights(N + K, N, K)
    q, s, z = spear.quantize_rtn(torch.from_numpy(w).cuda(), group_size)
    torch.cuda.synchronize()
    codes, s_ref, z_ref = rtn.rtn_quantize(w, group_size)
    np.testing.assert_array_equal(q.cpu().numpy(), rtn.pack_codes(codes))
    np.testing.assert_array_equal(s.cpu().view(torch.int16).numpy().view(np.uint16), s_ref)
    np.testing.assert_array_equal(z.cpu().numpy(), z_ref)


def test_rtn_rejects_bad_arguments():
    w = torch.zeros((4, 100), device="cuda")
    with pytest.raises(spear.SpearError):
        spear.quantize_rtn(w, 128)


def _quality(act_aware, gate, M=8):
    K = N = 1024
    rng = np.random.default_rng(5)
    W = torch.from_numpy(rng.normal(0, 0.02, size=(N, K)).astype(np.float32)).cuda()
    outl = wl.outlier_channels(K, 0, "rtn")
    xcal = wl.bf16_bits_to_f32(wl.make_x(K, 64, outl, 1, "rtn/cal")).astype(np.float64)
    a = torch.from_numpy(np.sqrt((xcal ** 2).mean(axis=0))).float().cuda() if act_aware else None
    q, s, z, A, B, wq = calibrate.quantize_and_init(W, 128, 64, a)
    x = wl.make_x(K, M, outl, 2, "rtn/x")
    y_fp = wl.bf16_bits_to_f32(x).astype(np.float64) @ W.double().cpu().numpy().T
    out = {}
    for name, (AA, BB) in {"w4": (None, None), "ec": (A, B)}.items():
        lin = spear.SpearLinear(K, N, 128, q, s, z, AA, BB, alpha=1.0, gate=gate, max_tokens=M)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        lin.forward_decode(dev_bf16(x), y)
        assert lin.check() == spear.SPEAR_OK
        out[name] = host_f64(y)
        lin.close()
    e = {k: np.linalg.norm(v - y_fp) / np.linalg.norm(y_fp) for k, v in out.items()}
    return e, (q, s, z, A, B, x, out)


def test_svd_init_through_the_kernel_matches_oracle_and_reduces_error():
    e, (q, s, z, A, B, x, out) = _quality(True, spear.SPEAR_GATE_ONE)
    # the compensated layer computed by the kernel matches the fp64 oracle on the same weights
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    yr = ref.forward(q.cpu().numpy(), bits(s), z.cpu().numpy(), 1024, 128, bits(A), bits(B), 1.0, 1, x)
    assert rel_err(out["ec"], yr) <= 1e-2
    # activation-aware static correction recovers most of the W4 output error
    assert e["ec"] < 0.6 * e["w4"], e
