"""The tensor-core GEMM engine on single problems, every variant the chain uses.

out = alpha * A op(B) + beta * aux + diag * I is compared with a float64 matmul of the
same bf16/fp16 inputs.  The only rounding on the GPU side is the final cast of the fp32
accumulator (plus the epilogue's fp32 arithmetic), so the bar is a few half-precision
ulps: relative Frobenius error <= 4e-3 for bf16 outputs and 5e-4 for fp16 outputs.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    m.lib()
    return m


def _rand(shape, dtype, seed):
    """Random matrix whose row stride is rounded up to 8 elements (a view when padded)."""
    rows, cols = shape
    ld = (cols + 7) // 8 * 8
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    full = torch.randn(rows, ld, generator=g, device="cuda").to(dtype)
    return full[:, :cols]


def _ref(a, b, aux, b_mn, alpha, beta, diag):
    A = a.double().cpu().numpy()
    B = b.double().cpu().numpy()
    prod = A @ (B if b_mn else B.T)
    out = alpha * prod
    if aux is not None:
        out = out + beta * aux.double().cpu().numpy()
    if diag:
        k = min(out.shape)
        out[np.arange(k), np.arange(k)] += diag
    return out


CASES = [
    # M, N, K, b_mn, aux, diag
    (128, 256, 64, False, False, 0.0),
    (128, 128, 128, False, False, 0.0),
    (256, 512, 1024, False, False, 0.0),
    (200, 136, 72, False, False, 0.0),
    (3, 5, 8, False, False, 0.0),
    (128, 256, 128, True, True, 0.0),
    (264, 328, 200, True, True, 0.0),
    (64, 1000, 64, True, False, 0.0),
    (192, 192, 192, False, True, 3.4445),
    (384, 384, 4096, False, True, 0.0),
    # the expert order of the Split/MoE table: the last column tile holds 128 of 256
    # columns, and the 2-SM kernel runs it as N = 128 MMAs (64 columns of B per CTA)
    (1408, 1408, 704, False, False, 0.0),
    (256, 1408, 512, True, True, 0.0),
    (272, 72, 136, True, False, 0.0),
]


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M,N,K,b_mn,use_aux,diag", CASES)
def test_gemm_variants(nsm, dtype, M, N, K, b_mn, use_aux, diag, pair):
    seed = M * 7 + N * 3 + K
    a = _rand((M, K), dtype, seed)
    b = _rand((K, N) if b_mn else (N, K), dtype, seed + 1)
    aux = _rand((M, N), dtype, seed + 2) if use_aux else None
    out = torch.full((M, (N + 7) // 8 * 8), float("nan"), dtype=dtype, device="cuda")[:, :N]
    alpha, beta = 0.75, -1.25
    nsm.gemm(a, b, out, aux, b_mn, alpha, beta, diag, pair=pair)
    assert nsm.device_status() == nsm.NSM_OK
    ref = _ref(a, b, aux, b_mn, alpha, beta if use_aux else 0.0, diag)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    tol = 4e-3 if dtype == torch.bfloat16 else 5e-4
    assert rel <= tol, rel


def test_gemm_padded_leading_dimension(nsm):
    # operands that are views into wider buffers (row stride > row length)
    M, N, K = 160, 200, 96
    a_full = _rand((M, K + 32), torch.bfloat16, 1)
    b_full = _rand((N, K + 64), torch.bfloat16, 2)
    out_full = torch.zeros((M, N + 56), dtype=torch.bfloat16, device="cuda")
    a, b, out = a_full[:, :K], b_full[:, :K], out_full[:, :N]
    nsm.gemm(a, b, out)
    torch.cuda.synchronize()
    ref = _ref(a, b, None, False, 1.0, 0.0, 0.0)
    rel = np.linalg.norm(out.double().cpu().numpy() - ref) / np.linalg.norm(ref)
    assert rel <= 4e-3
    # columns beyond N untouched
    assert torch.count_nonzero(out_full[:, N:]).item() == 0


@pytest.mark.parametrize("pair", [False, True])
def test_gemm_deterministic(nsm, pair):
    a = _rand((512, 2048), torch.bfloat16, 5)
    o1 = torch.empty((512, 512), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    nsm.gemm(a, a, o1, pair=pair)
    nsm.gemm(a, a, o2, pair=pair)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("b_mn", [False, True])
def test_gemm_pair_matches_single_cta(nsm, dtype, b_mn):
    # the two kernels accumulate each output over K in the same order of 16-wide MMAs
    # into fp32 TMEM and round once in the same epilogue: the results are the same bits
    a = _rand((768, 1536), dtype, 8)
    b = _rand((1536, 1016) if b_mn else (1016, 1536), dtype, 9)
    aux = _rand((768, 1016), dtype, 10)
    o1 = torch.empty((768, 1016), dtype=dtype, device="cuda")
    o2 = torch.empty_like(o1)
    nsm.gemm(a, b, o1, aux=aux, b_mn_major=b_mn, alpha=0.75, beta=-1.5, pair=False)
    nsm.gemm(a, b, o2, aux=aux, b_mn_major=b_mn, alpha=0.75, beta=-1.5, pair=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    # and a symmetric output, upper tiles mirrored
    s1 = torch.empty((768, 768), dtype=dtype, device="cuda")
    s2 = torch.empty_like(s1)
    nsm.gemm(a, a, s1, symmetric=True, pair=False)
    nsm.gemm(a, a, s2, symmetric=True, pair=True)
    torch.cuda.synchronize()
    assert torch.equal(s1, s2)


def test_gemm_rejects_bad_arguments(nsm):
    a = torch.zeros((16, 12), dtype=torch.bfloat16, device="cuda")  # row stride 12
    b = torch.zeros((16, 12), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nsm.NsmError) as e:
        nsm.gemm(a, b, out)
    assert e.value.code == nsm.NSM_ERR_ALIGN


SYM_CASES = [(128, 64), (200, 72), (256, 256), (384, 1024), (1000, 136), (64, 64), (3, 8), (520, 4096),
             (1408, 2048)]


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M,K", SYM_CASES)
@pytest.mark.parametrize("use_aux", [False, True])
def test_gemm_symmetric_output(nsm, dtype, M, K, use_aux, pair):
    # A A^T (+ beta S + diag I with S symmetric) computed on the upper-triangle tiles only
    seed = M * 11 + K
    a = _rand((M, K), dtype, seed)
    aux = None
    if use_aux:
        s = _rand((M, M), torch.float32, seed + 1)
        s = (s + s.T).to(dtype)
        ld = (M + 7) // 8 * 8
        aux = torch.zeros((M, ld), dtype=dtype, device="cuda")[:, :M]
        aux.copy_(s)
    ld = (M + 7) // 8 * 8
    out_full = torch.full((M, ld + 8), float("nan"), dtype=dtype, device="cuda")
    out = out_full[:, :M]
    alpha, beta, diag = 0.5, -1.5, (2.0 if use_aux else 0.0)
    nsm.gemm(a, a, out, aux, False, alpha, beta, diag, symmetric=True, pair=pair)
    assert nsm.device_status() == nsm.NSM_OK
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, got.T)  # exactly symmetric
    ref = _ref(a, a, aux, False, alpha, beta if use_aux else 0.0, diag)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= (4e-3 if dtype == torch.bfloat16 else 5e-4), rel
    # nothing written past the M columns of the view
    assert torch.isnan(out_full[:, M:ld].float()).all() if ld > M else True
    assert torch.isnan(out_full[:, ld:].float()).all()


def test_gemm_symmetric_rejects_rectangular(nsm):
    a = _rand((64, 64), torch.bfloat16, 0)
    b = _rand((128, 64), torch.bfloat16, 1)
    out = torch.empty((64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nsm.NsmError) as e:
        nsm.gemm(a, b, out, symmetric=True)
    assert e.value.code == nsm.NSM_ERR_SHAPE
