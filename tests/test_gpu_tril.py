"""GPU parity of gdn_unit_lower_inverse -- the intra-chunk (I + A)^-1 by forward
substitution and by the Neumann product -- against the oracle's fp64 forward
substitution (itself pinned by T (I + A) = I and the finite Neumann series).
Tolerances (relative Frobenius): substitution (fp32) 1e-5; Neumann (tf32 operands,
fp32 accumulation, six rounds) 5e-3."""
import numpy as np
import pytest
import torch

from gpu_util import DEV, ensure_built, rel
import oracle
import linear_attention_recurrence_03_gb300 as gdn

pytestmark = pytest.mark.gpu
TOL = {gdn.GDN_TRIL_SUBSTITUTION: 1e-5, gdn.GDN_TRIL_NEUMANN: 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def chunk_A(n, seed=0, C=64, Dk=128):
    """A[r, j] = beta_r (k_r . k_j) exp(gamma_r - gamma_j) for j < r: the strictly lower
    matrix of a chunk, from unit keys, beta ~ U(0.05, 0.95), g ~ U(-0.3, -0.005)."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n, C, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    beta = rng.uniform(0.05, 0.95, (n, C))
    gam = np.cumsum(rng.uniform(-0.3, -0.005, (n, C)), axis=1)
    A = beta[:, :, None] * np.einsum("nrd,njd->nrj", k, k) * np.exp(gam[:, :, None] - gam[:, None, :])
    return np.tril(A, -1).astype(np.float32)


@pytest.mark.parametrize("alg", [gdn.GDN_TRIL_SUBSTITUTION, gdn.GDN_TRIL_NEUMANN])
def test_unit_lower_inverse_matches_oracle(alg):
    A = chunk_A(37)
    T = gdn.gdn_unit_lower_inverse(torch.from_numpy(A).to(DEV), alg).cpu().numpy()
    for i in (0, 18, 36):
        ref = oracle.unit_lower_inverse(A[i])
        assert rel(T[i], ref) <= TOL[alg], f"matrix {i}"
        assert np.all(np.triu(T[i], 1) == 0) and np.all(np.diag(T[i]) == 1)
    err = max(rel(T[i] @ (np.eye(64) + A[i]), np.eye(64)) for i in range(37))
    assert err <= 10 * TOL[alg]


def test_unit_lower_inverse_in_place_and_algorithms_agree():
    A = chunk_A(8, seed=3)
    a = torch.from_numpy(A).to(DEV)
    t_sub = gdn.gdn_unit_lower_inverse(a, gdn.GDN_TRIL_SUBSTITUTION)
    t_neu = gdn.gdn_unit_lower_inverse(a, gdn.GDN_TRIL_NEUMANN)
    b = a.clone()
    gdn.gdn_unit_lower_inverse(b, gdn.GDN_TRIL_SUBSTITUTION, out=b)
    torch.cuda.synchronize()
    assert torch.equal(b, t_sub)
    assert rel(t_neu.cpu().numpy(), t_sub.cpu().numpy()) <= TOL[gdn.GDN_TRIL_NEUMANN]
