"""csr_validate on the GPU against the oracle's CSR check (the code of the
first violation) and a numpy restatement of the rule order (its index).

Every malformed case below keeps the arrays exactly as long as the sizes
passed (row_offsets M+1, col_indices nnz): the kernel reads offsets at r and
r+1 < M+1 and entries only inside [0, nnz) after clamping, so planted
violations are reported, never followed."""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

# oracle_csr_check's negative codes -> usm_csr_check codes
ORACLE_TO_CODE = {0: 0, -2: 1, -3: 2, -4: 3, -5: 4, -6: 5}


def expected(M, K, ro, ci):
    """(code, index) from the rule order written out with numpy."""
    ro, ci = np.asarray(ro, np.int64), np.asarray(ci, np.int64)
    nnz = ci.size
    if ro[0] != 0:
        return 1, 0
    dec = np.nonzero(ro[1:] < ro[:-1])[0]
    if dec.size:
        return 2, int(dec[0])
    if ro[M] != nnz:
        return 3, M
    rows = np.repeat(np.arange(M), np.diff(ro))
    pos = np.arange(nnz)
    bad_range = (ci < 0) | (ci >= K)
    prev = np.concatenate([[np.iinfo(np.int64).min], ci[:-1]])
    bad_order = (pos > ro[rows]) & (ci <= prev)
    bad = np.nonzero(bad_range | bad_order)[0]
    if not bad.size:
        return 0, -1
    p = int(bad[0])
    return (4 if bad_range[p] else 5), p


def base_csr():
    csr = W.random_csr([300, 200, 77], 300, 200, 0.1)
    return 300, 200, csr.row_offsets.copy(), csr.col_indices.copy()


def planted():
    M, K, ro, ci = base_csr()
    row_with = [r for r in range(M) if ro[r + 1] - ro[r] >= 3]
    r1, r2 = row_with[3], row_with[-2]
    cases = {"valid": (M, K, ro, ci)}

    def case(name, ro_=None, ci_=None):
        cases[name] = (M, K, ro if ro_ is None else ro_, ci if ci_ is None else ci_)

    x = ro.copy(); x[0] = 1; case("first_offset", ro_=x)
    x = ro.copy(); x[0] = -7; case("first_offset_negative", ro_=x)
    x = ro.copy(); x[150] = x[151] + 2; case("decrease_mid", ro_=x)
    x = ro.copy(); x[M - 1] = x[M] + 5; case("decrease_last_row", ro_=x)
    x = ro.copy(); x[M] -= 3; case("last_offset_short", ro_=x)
    x = ro.copy(); x[M] = 2**31 - 1; x[M - 1] = min(x[M - 1], x[M]); case("last_offset_huge", ro_=x)
    y = ci.copy(); y[ro[r1] + 1] = K; case("column_equal_K", ci_=y)
    y = ci.copy(); y[ro[r2]] = -1; case("column_negative", ci_=y)
    y = ci.copy(); y[ro[r1] + 2] = y[ro[r1] + 1]; case("column_duplicate", ci_=y)
    y = ci.copy(); y[ro[r2] + 1], y[ro[r2] + 2] = y[ro[r2] + 2], y[ro[r2] + 1]; case("column_swapped", ci_=y)
    y = ci.copy(); y[ro[r1] + 1] = y[ro[r1]]; y[ro[r2]] = K + 9; case("order_before_range", ci_=y)
    y = ci.copy(); y[ro[r1] + 1] = K + 1; y[ro[r2] + 1] = y[ro[r2]]; case("range_before_order", ci_=y)
    y = ci.copy(); y[ro[r1] + 1] = -3; case("both_at_one_position", ci_=y)
    # a row start below its predecessor's last column is fine (order is per row)
    y = ci.copy(); y[ro[r1]] = 0; y[ro[r1] - 1] = K - 1; case("row_boundary_not_order", ci_=y)
    x = ro.copy(); x[0] = 3; x[150] = x[151] + 2; y = ci.copy(); y[5] = K
    case("offsets_win_over_columns", ro_=x, ci_=y)
    return cases


@pytest.mark.parametrize("name", sorted(planted()))
def test_validate_matches_oracle(usm, name):
    M, K, ro, ci = planted()[name]
    ro = np.asarray(ro, np.int32)
    ci = np.asarray(ci, np.int32)
    code, index = usm.csr_validate(dev(ro), dev(ci), K)
    assert (code, index) == expected(M, K, ro, ci), name
    assert code == ORACLE_TO_CODE[oracle.csr_check(M, K, ro, ci)], name
    assert (code == 0) == (name in ("valid", "row_boundary_not_order"))


def test_validate_empty_and_tiny(usm):
    e = np.zeros(0, np.int32)
    assert usm.csr_validate(dev(np.zeros(1, np.int32)), dev(e), 4) == (0, -1)    # M = 0
    assert usm.csr_validate(dev(np.zeros(4, np.int32)), dev(e), 4) == (0, -1)    # empty rows
    assert usm.csr_validate(dev(np.array([0, 0, 1], np.int32)), dev(e), 4) == (3, 2)  # claims a nonzero
    assert usm.csr_validate(dev(np.array([0, 1], np.int32)), dev(np.array([4], np.int32)), 4) == (4, 0)
    assert usm.csr_validate(dev(np.array([0, 1], np.int32)), dev(np.array([3], np.int32)), 4) == (0, -1)


def test_validate_workload_matrices(usm):
    """The seeded workloads (full sizes) satisfy the contract."""
    for p in [W.tiny(), W.ffn(4096, 1024, 70, with_sddmm=False), W.lstm(50), W.attention()]:
        csr = p.csr
        K = int(csr.K)
        got = usm.csr_validate(dev(csr.row_offsets), dev(csr.col_indices), K)
        assert got == (0, -1), p.name


def dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()
