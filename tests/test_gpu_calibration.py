"""GPU parity of the device-side calibration (oscar_calibration_covariances):
the covariance targets of the rotations, "OSCAR: Offline Spectral
Covariance-Aware Rotation ..." (gist.science, it), Riepilogo Tecnico 2.2 A,

  C_Q = (1/(N g)) sum_j Q_j^T Q_j,  C_S = (1/(N g)) sum_j (S_j V)^T (S_j V),

against the float64 oracle (relative Frobenius error within float32
accumulation, 2e-5), the rotations built from them on the host against the
oracle's covariances (they diagonalise them, eigenvalues descending), and a
layer calibrated this way through the whole write and read path."""

import numpy as np
import pytest
import torch

import oracle
from bit_rotated_kv_oscar_gb300 import abi, build
from bit_rotated_kv_oscar_gb300.calibrate import calibrate_device
from synth import draw_kv, draw_queries
from tests.gpu_harness import D, Layer
from tests.test_gpu_parity import check_decode, check_int2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    build.build()
    abi.lib()


def calib_data(seed, n, hq, hkv, spikes=False):
    q = draw_queries(seed, 900, n, hq, hkv, D).numpy()
    k, v = (t.numpy() for t in draw_kv(seed, 900, n, hkv, D, spikes))
    return q, k, v


def oracle_covariances(q, k, v):
    n, hq, _ = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    scale = 1.0 / np.sqrt(D)
    c_q = np.zeros((hkv, D, D))
    c_s = np.zeros((hkv, D, D))
    for h in range(hkv):
        for j in range(h * g, (h + 1) * g):
            c_q[h] += oracle.query_covariance(q[:, j]) / g
            c_s[h] += oracle.score_weighted_value_covariance(q[:, j], k[:, h], v[:, h], scale) / g
    return c_q, c_s


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("hq,hkv,n", [(32, 8, 512), (8, 2, 1000), (64, 8, 300), (4, 4, 65)])
def test_covariances_match_the_oracle(hq, hkv, n):
    q, k, v = calib_data(hq + n, n, hq, hkv)
    dev = lambda a: torch.as_tensor(a).to("cuda", torch.bfloat16).contiguous()  # noqa: E731
    c_q, c_s = abi.calibration_covariances(dev(q), dev(k), dev(v))
    torch.cuda.synchronize()
    ref_q, ref_s = oracle_covariances(q, k, v)
    for h in range(hkv):
        assert rel_fro(c_q[h].cpu().numpy(), ref_q[h]) <= 2e-5, h
        assert rel_fro(c_s[h].cpu().numpy(), ref_s[h]) <= 2e-5, h
        assert np.allclose(c_q[h].cpu().numpy(), c_q[h].cpu().numpy().T, rtol=0, atol=1e-6 * np.abs(ref_q[h]).max())


def test_rotations_diagonalise_the_oracle_covariances():
    q, k, v = calib_data(3, 1024, 32, 8)
    d = calibrate_device(q, k, v)
    ref_q, ref_s = oracle_covariances(q, k, v)
    hp = oracle.hadamard(D) @ oracle.bit_reversal_matrix(D)
    for r, c in ((d["R_K"], ref_q), (d["R_V"], ref_s)):
        for h in range(r.shape[0]):
            rh = r[h].astype(np.float64)
            assert np.abs(rh.T @ rh - np.eye(D)).max() <= 1e-5
            u = rh @ hp.T                           # R = U H P, H P orthogonal
            m = u.T @ c[h] @ u
            off = m - np.diag(np.diag(m))
            assert np.linalg.norm(off) <= 1e-4 * np.linalg.norm(c[h]), h
            diag = np.diag(m)
            assert np.all(np.diff(diag) <= 1e-5 * diag[0]), h   # descending


@pytest.mark.parametrize("group", [32, 64])
def test_device_calibrated_layer_round_trip(group):
    layer = Layer(32, 8, 4, 128, 2, 3000, seed=23, device_calibration=True, group=group)
    trace = layer.new_trace(3000)
    k, v = layer.draw(2500)
    layer.append(0, k, v, trace)
    k, v = layer.draw(900)
    layer.append(1, k, v)
    check_int2(layer, 0, trace)
    check_decode(layer, 2)
    assert layer.ctx.error_flags() == 0


def test_workspace_and_arguments_are_checked():
    q = torch.zeros(10, 4, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(10, 2, D, dtype=torch.bfloat16, device="cuda")
    need = abi.lib().oscar_calibration_workspace_bytes(10, 4)
    assert need == 4 * 10 * D * 4
    ws = torch.empty(need // 4 - 1, dtype=torch.float32, device="cuda")
    c = torch.empty(2, D, D, dtype=torch.float32, device="cuda")
    st = abi.lib().oscar_calibration_covariances(abi._ptr(q), abi._ptr(k), abi._ptr(k), 10, 4, 2, 0.0,
                                                 abi._ptr(c), abi._ptr(c), abi._ptr(ws), need - 4, None)
    assert st == -3  # workspace one float short: OSCAR_ERR_OUT_OF_RANGE
    st = abi.lib().oscar_calibration_covariances(abi._ptr(q), abi._ptr(k), abi._ptr(k), 10, 3, 2, 0.0,
                                                 abi._ptr(c), abi._ptr(c), abi._ptr(ws), need, None)
    assert st == -1  # 3 query heads over 2 KV heads: OSCAR_ERR_INVALID_ARG
