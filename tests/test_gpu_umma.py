"""The tensor-core fold building block (tcgen05.mma into tensor memory) against a
float64 matrix product: D = A[:, :w+1] @ B[:w+1] for 128 rows, with A float32 carried
by three bf16 parts and B bf16 in the ring layout. This pins the shared-memory
operand layouts, the instruction descriptor and the tensor-memory lane layout the
decode kernels' flush folds use.

Tolerance: the three-part split carries A's float32 significand, the products of
bf16 parts are exact, and the tensor core accumulates in float32, so the error is a
few float32 roundings of the sum of |terms|: |D - ref| <= 2^-20 * (|A| @ |B|)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    import ssm_linear_attention_gb300 as ssm
    ssm.lib()


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("N", [128, 64])
@pytest.mark.parametrize("w", [15, 0, 6])
def test_umma_fold_matches_float64_product(N, w):
    import ssm_linear_attention_gb300 as ssm
    r = np.random.default_rng(100 + 7 * w + N)
    # coefficients spanning several binades, as decay products times dt times x do
    A = (r.standard_normal((128, 16)) * np.exp(r.uniform(-6, 2, (128, 16)))).astype(np.float32)
    Bb = _bf16(r.standard_normal((16, N)) / np.sqrt(128))
    B = Bb.float().numpy().astype(np.float64)
    D = torch.full((128, N), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssm.rssm_debug_umma_fold(torch.from_numpy(A).cuda(), Bb.view(torch.int16).cuda(), w, N, D, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = D.cpu().numpy().astype(np.float64)
    A64 = A.astype(np.float64)
    ref = A64[:, : w + 1] @ B[: w + 1]
    bound = 2.0 ** -20 * (np.abs(A64[:, : w + 1]) @ np.abs(B[: w + 1])) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


def test_umma_fold_ignores_entries_above_w():
    import ssm_linear_attention_gb300 as ssm
    r = np.random.default_rng(5)
    A = r.standard_normal((128, 16)).astype(np.float32)
    A[:, 4:] = np.nan                         # entries above w are never read as operands
    Braw = r.standard_normal((16, 128)).astype(np.float32)
    Braw[4:] = np.inf
    Bb = _bf16(Braw)
    D = torch.zeros(128, 128, device="cuda")
    ssm.rssm_debug_umma_fold(torch.from_numpy(A).cuda(), Bb.view(torch.int16).cuda(), 3, 128, D)
    torch.cuda.synchronize()
    ref = A[:, :4].astype(np.float64) @ Bb.float().numpy()[:4].astype(np.float64)
    assert np.all(np.isfinite(D.cpu().numpy()))
    assert np.allclose(D.cpu().numpy(), ref, rtol=1e-5, atol=1e-6)
