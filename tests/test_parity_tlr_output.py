"""GPU parity of the TLR-output path against the oracle's recompression.

``tlr_compress`` turns the tiles of a dense matrix into TLR form ("TLR Matrix
Multiplication", section "Introduction: TLR GEMM": the TLR-output cases; the
truncation rule is this build's reading, written out in oracle/tlr_output.py).
The oracle takes each tile's exact SVD in fp64; the GPU sketches the tile with a
Gaussian matrix passed in as an input, so it reproduces the truncated SVD when
the sketch holds the tile's range (s >= the tile's numerical rank, always when
s >= b). The comparisons:

* ranks equal to the oracle's wherever the oracle's decision is not within 5 %
  of the threshold (there either neighbouring rank is correct);
* every tile's U V^T within the stated tolerance of the oracle's U V^T when the
  ranks agree, and of the tile itself within eps (the rule's bound);
* the reported error equal to the measured one;
* for a product (dense-output product on TF32 tensor cores, then the
  recompression) the oracle's product and recompression, at the fp32 tolerance
  of the dense path (2e-3), and the packed result read back by ``tlr_gemm``.
"""
import numpy as np
import pytest

import oracle
import tlr_inputs as ti
from oracle import tlr_output as to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


@pytest.fixture(scope="module")
def handle(torch_cuda):
    import gemm_tlr_gb300 as g
    h = g.tlr_create(torch_cuda.cuda.current_stream().cuda_stream)
    yield h
    g.tlr_destroy(h)


def _upload(torch, M):
    return torch.from_numpy(np.asfortranarray(M, dtype=np.float32).reshape(-1, order="F")).cuda()


def _compress(torch, handle, M, b, dense_diag, eps, r_max, s, seed=0, batch_tiles=None):
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300.device import DeviceCompression
    m, n = M.shape
    C = _upload(torch, M)
    dc = DeviceCompression(m, n, b, dense_diag, eps, r_max, ti.sketch(b, s, seed), batch_tiles=batch_tiles)
    dc.run(handle, C, m)
    assert g.tlr_get_device_status(handle) == 0
    return dc, dc.tiles()


def _oracle(M, b, dense_diag, eps, r_max):
    """The oracle's recompression of the same fp32 values, tile by tile."""
    M = np.asarray(M, dtype=np.float32).astype(np.float64)
    m, n = M.shape
    out = {}
    for i in range(-(-m // b)):
        for j in range(-(-n // b)):
            T = M[i * b:(i + 1) * b, j * b:(j + 1) * b]
            if dense_diag and i == j:
                out[(i, j)] = ("dense", T)
                continue
            U, V, r, err = to.compress_tile(T, eps, min(r_max, *T.shape))
            sig = np.linalg.svd(T, compute_uv=False)
            out[(i, j)] = ("lr", U, V, r, err, sig)
    return out


# The GPU keeps tile energies to about 1e-5 of the tile's (fp32 products and
# eigenvalues): squared relative errors are compared with this slack.
E2 = 2e-5


def _near_tie(sig, r, eps, r_cap):
    """True when rank r's decision is within reach of the GPU's energy precision:
    a squared tail within 10 % (plus E2) of eps^2 on either side of r."""
    tot = np.sum(sig ** 2)
    if tot == 0:
        return False
    tail2 = lambda k: np.sum(sig[k:] ** 2) / tot
    close = lambda k: abs(tail2(k) - eps ** 2) <= 0.1 * eps ** 2 + E2
    return close(r) or (r > 0 and close(r - 1)) or r >= r_cap


def _compare(gpu, ora, M, eps, tol_uv, r_cap, allow_tie=True):
    """Per-tile comparison; returns the number of tiles whose ranks matched."""
    M = np.asarray(M, dtype=np.float32).astype(np.float64)
    b_r, b_c = gpu["rdims"], gpu["cdims"]
    r0 = np.concatenate([[0], np.cumsum(b_r)])
    c0 = np.concatenate([[0], np.cumsum(b_c)])
    matched = 0
    for (i, j), o in ora.items():
        T = M[r0[i]:r0[i + 1], c0[j]:c0[j + 1]]
        kind, *f = gpu["tiles"][(i, j)]
        if o[0] == "dense":
            assert kind == "dense"
            assert np.array_equal(f[0], T), (i, j)            # copied, bit for bit
            continue
        _, Uo, Vo, ro, erro, sig = o
        Ug, Vg = f
        rg = int(gpu["ranks"][i, j])
        nrm = np.linalg.norm(T)
        approx = Ug @ Vg.T
        measured = np.linalg.norm(T - approx) / nrm if nrm > 0 else 0.0
        # the reported error is the measured one, and within eps unless capped
        eg = gpu["errors"][i, j]
        assert abs(eg ** 2 - measured ** 2) <= E2 + 2e-3 * measured ** 2, (i, j, eg, measured)
        cap = min(r_cap, *T.shape)
        if rg < cap:
            assert measured ** 2 <= eps ** 2 + E2, (i, j, measured, eps)
        if rg == ro:
            matched += 1
            ref = Uo @ Vo.T
            d = np.linalg.norm(approx - ref) / max(np.linalg.norm(ref), 1e-30)
            assert d <= tol_uv, (i, j, rg, d)
        else:
            assert allow_tie and _near_tie(sig, ro, eps, cap) and abs(rg - ro) <= 1, (i, j, rg, ro)
    return matched


def _spectrum_tile(rng, n, sigma):
    q1, _ = np.linalg.qr(rng.standard_normal((n, n)))
    q2, _ = np.linalg.qr(rng.standard_normal((n, n)))
    s = np.zeros(n)
    s[:len(sigma)] = sigma
    return q1 @ np.diag(s) @ q2.T


@pytest.mark.parametrize("b", [64, 128, 10])
@pytest.mark.parametrize("eps", [0.3, 0.1, 0.03, 0.01])
def test_prescribed_spectra(torch_cuda, handle, eps, b):
    """Tiles with singular values base^-k (a different base per tile): the
    sketch spans each tile (s = b), so ranks and factors are the oracle's.
    b = 128 runs the Jacobi kernel compiled for 128-column sketches, b = 64
    and b = 10 (five pairs of rows) the general one."""
    rng = np.random.default_rng(11)
    nt = 3
    M = np.zeros((b * nt, b * nt))
    for i in range(nt):
        for j in range(nt):
            base = 1.3 + 0.25 * (i * nt + j)
            M[i * b:(i + 1) * b, j * b:(j + 1) * b] = _spectrum_tile(rng, b, [base ** -k for k in range(b)])
    _, gpu = _compress(torch_cuda, handle, M, b, False, eps, b, b)
    ora = _oracle(M, b, False, eps, b)
    assert _compare(gpu, ora, M, eps, 2e-4, b) >= nt * nt - 1


def test_exact_low_rank_tiles_with_a_small_sketch(torch_cuda, handle):
    """Tiles of exact rank r <= 20 with b = 128 and s = 32: the sketch holds the
    range, ranks equal r and U V^T is the tile."""
    rng = np.random.default_rng(12)
    b, nt = 128, 3
    R = rng.integers(0, 21, size=(nt, nt))
    M = np.zeros((b * nt, b * nt))
    for i in range(nt):
        for j in range(nt):
            r = R[i, j]
            M[i * b:(i + 1) * b, j * b:(j + 1) * b] = rng.standard_normal((b, r)) @ rng.standard_normal((r, b))
    _, gpu = _compress(torch_cuda, handle, M, b, False, 1e-2, 32, 32)
    ora = _oracle(M, b, False, 1e-2, 32)
    for (i, j), o in ora.items():
        assert o[3] == R[i, j]
    assert _compare(gpu, ora, M, 1e-2, 1e-4, 32, allow_tie=False) == nt * nt
    assert (gpu["ranks"] == R).all()


def test_rank_cap_reports_the_larger_error(torch_cuda, handle):
    """Full-rank tiles with a flat spectrum, r_max = 8, s = 16: both sides keep
    8; the sketched factors are close to optimal and report their own error."""
    rng = np.random.default_rng(13)
    b = 64
    M = rng.standard_normal((2 * b, 2 * b))
    _, gpu = _compress(torch_cuda, handle, M, b, False, 1e-3, 8, 16)
    ora = _oracle(M, b, False, 1e-3, 8)
    for (i, j), o in ora.items():
        assert o[3] == 8 and gpu["ranks"][i, j] == 8
        err_opt = o[4]
        assert err_opt - 1e-5 <= gpu["errors"][i, j] <= 1.5 * err_opt, (gpu["errors"][i, j], err_opt)


@pytest.mark.parametrize("batch_tiles", [None, 3])
def test_ragged_tiles_and_dense_diagonal(torch_cuda, handle, batch_tiles):
    """N = 200, b = 64: a ragged last tile row and column (8 wide), dense
    diagonal tiles copied as they are; the same result with the tiles run in
    batches of three (a smaller workspace)."""
    rng = np.random.default_rng(14)
    n, b = 200, 64
    dims = ti.tile_dims(n, b)
    off = np.concatenate([[0], np.cumsum(dims)])
    M = np.zeros((n, n))
    for i, di in enumerate(dims):
        for j, dj in enumerate(dims):
            if i == j:
                M[off[i]:off[i + 1], off[j]:off[j + 1]] = rng.standard_normal((di, dj))
            else:
                r = min(int(rng.integers(0, 7)), di, dj)
                M[off[i]:off[i + 1], off[j]:off[j + 1]] = rng.standard_normal((di, r)) @ rng.standard_normal((r, dj))
    _, gpu = _compress(torch_cuda, handle, M, b, True, 1e-2, 16, 16, batch_tiles=batch_tiles)
    ora = _oracle(M, b, True, 1e-2, 16)
    assert _compare(gpu, ora, M, 1e-2, 1e-4, 16) >= len(dims) * (len(dims) - 1) - 1


def _identity(n, b):
    """The identity as a TLR matrix: identity diagonal tiles (and corner), rank-0 tiles elsewhere."""
    nt, mf, rem = -(-n // b), n // b, n % b
    I = ti.make_tlr(np.random.default_rng(0), n, b, None, "f32", ranks=np.zeros((nt, nt), dtype=np.int64))
    for t in range(mf):
        I.D[t * b * b:(t + 1) * b * b] = np.eye(b, dtype=np.float32).reshape(-1, order="F")
    if rem:
        I.gamma[:] = np.eye(rem, dtype=np.float32).reshape(-1, order="F")
    return I


def _product_then_compress(torch, handle, p, eps, r_max, s):
    from gemm_tlr_gb300.device import DeviceProblem
    import gemm_tlr_gb300 as g
    dp = DeviceProblem(p)
    try:
        dp.make_plan(handle)
        dp.reset_c()
        dp.run()
        assert g.tlr_get_device_status(handle) == 0
        from gemm_tlr_gb300.device import DeviceCompression
        b = p.A.b
        dense_diag = p.m == p.n and p.A.diag_dense and p.B.diag_dense
        dc = DeviceCompression(p.m, p.n, b, dense_diag, eps, r_max, ti.sketch(b, s))
        dc.run(handle, dp.C, dp.ldc)
        assert g.tlr_get_device_status(handle) == 0
        return dc, dc.tiles(), dp.result()
    finally:
        dp.close()


def _compare_product(gpu, ora, C, eps, tol, r_cap):
    """TLR-output product against the oracle's (C: the oracle's dense product).
    Per tile: the GPU's U V^T is as close to the exact tile as the error it
    reports, up to the dense path's own tolerance; that error is within eps
    unless the rank is capped; where the ranks agree the errors agree within
    tol, and where they differ the oracle's decision is within 5 % of the
    threshold. Returns the number of low-rank tiles whose ranks agree."""
    r0 = np.concatenate([[0], np.cumsum(gpu["rdims"])])
    c0 = np.concatenate([[0], np.cumsum(gpu["cdims"])])
    agree = 0
    for (i, j), o in ora["tiles"].items():
        T = C[r0[i]:r0[i + 1], c0[j]:c0[j + 1]]
        nrm = max(np.linalg.norm(T), 1e-30)
        kind, *f = gpu["tiles"][(i, j)]
        if o[0] == "dense":
            assert kind == "dense" and np.linalg.norm(f[0] - T) / nrm <= tol, (i, j)
            continue
        rg, ro = int(gpu["ranks"][i, j]), int(ora["ranks"][i, j])
        eg, eo = gpu["errors"][i, j], ora["errors"][i, j]
        e_true = np.linalg.norm(f[0] @ f[1].T - T) / nrm
        assert e_true <= np.sqrt(eg ** 2 + E2) + tol, (i, j, e_true, eg)
        cap = min(r_cap, *T.shape)
        if rg < cap:
            assert eg ** 2 <= eps ** 2 + E2, (i, j, eg)
        if rg == ro:
            agree += 1
            assert abs(eg - eo) <= tol + np.sqrt(E2), (i, j, eg, eo)
        else:
            sig = np.linalg.svd(T, compute_uv=False)
            assert abs(rg - ro) <= 1 and _near_tie(sig, ro, eps, cap), (i, j, rg, ro)
    return agree


def test_product_times_identity_recovers_the_operand(torch_cuda, handle):
    """A I through the dense-output product (TF32) and the recompression: every
    off-diagonal tile keeps A's rank, as in the oracle's pin."""
    rng = np.random.default_rng(3)
    n, b = 384, 64
    A = ti.make_tlr(rng, n, b, ti.rank_uniform(0, 12), "f32")
    p = ti.Problem("times_identity", A, _identity(n, b), "N", "N", 1.0, 0.0, None, n, n, "f32")
    _, gpu, _ = _product_then_compress(torch_cuda, handle, p, 1e-2, 32, 32)
    ora = to.tlr_output_product(p, 1e-2, 32)
    nt = n // b
    off = ~np.eye(nt, dtype=bool)
    assert (ora["ranks"][off] == A.ranks[off]).all()
    assert (gpu["ranks"][off] == A.ranks[off]).all()
    assert _compare_product(gpu, ora, oracle.gemm_problem(p), 1e-2, 2e-3, 32) == nt * (nt - 1)


def test_beta_term_joins_the_compressed_tile(torch_cuda, handle):
    """A I + 0.5 C0 with a rank-one C0: the ranks are the oracle's (r_ik + 1
    wherever its decision is clear)."""
    rng = np.random.default_rng(4)
    n, b = 256, 64
    A = ti.make_tlr(rng, n, b, ti.rank_uniform(1, 8), "f32")
    x, y = rng.standard_normal(n), rng.standard_normal(n)
    C0 = np.outer(x, y).astype(np.float32).reshape(-1, order="F")
    p = ti.Problem("a_plus_rank_one", A, _identity(n, b), "N", "N", 1.0, 0.5, C0, n, n, "f32")
    _, gpu, _ = _product_then_compress(torch_cuda, handle, p, 1e-2, 16, 16)
    ora = to.tlr_output_product(p, 1e-2, 16)
    nt = n // b
    assert _compare_product(gpu, ora, oracle.gemm_problem(p), 1e-2, 2e-3, 16) >= nt * (nt - 1) - 1


@pytest.mark.parametrize("eps", [0.1, 0.02])
def test_tiny_fixed_rank_product(torch_cuda, handle, eps):
    """The tiny fixed-rank TLR x TLR product (N = 512, b = 64, rank 8, fp32)
    with TLR output; s = b, so the sketch spans every tile."""
    p = ti.problem(1)
    _, gpu, _ = _product_then_compress(torch_cuda, handle, p, eps, 64, 64)
    ora = to.tlr_output_product(p, eps, 64)
    agree = _compare_product(gpu, ora, oracle.gemm_problem(p), eps, 2e-3, 64)
    assert agree >= 0.8 * 8 * 7


def _pack_numpy(tiles, ranks, n, b):
    """The packed format of include/tlr_gemm.h written out from the per-tile
    factors (interior U by tile row, V by tile column, D; boundary panels)."""
    mf, rem = n // b, n % b
    U, V, D = [], [], []
    for i in range(mf):
        for k in range(mf):
            if i != k and ranks[i, k] > 0:
                U.append(tiles[(i, k)][1].reshape(-1, order="F"))
    for k in range(mf):
        for i in range(mf):
            if i != k and ranks[i, k] > 0:
                V.append(tiles[(i, k)][2].reshape(-1, order="F"))
    for t in range(mf):
        D.append(tiles[(t, t)][1].reshape(-1, order="F"))
    out = {"U": U, "V": V, "D": D}
    if rem:
        out["bu_U"] = [tiles[(i, mf)][1].reshape(-1, order="F") for i in range(mf) if ranks[i, mf] > 0]
        out["bu_V"] = [tiles[(i, mf)][2].reshape(-1, order="F") for i in range(mf) if ranks[i, mf] > 0]
        out["bv_U"] = [tiles[(mf, j)][1].reshape(-1, order="F") for j in range(mf) if ranks[mf, j] > 0]
        out["bv_V"] = [tiles[(mf, j)][2].reshape(-1, order="F") for j in range(mf) if ranks[mf, j] > 0]
        out["gamma"] = [tiles[(mf, mf)][1].reshape(-1, order="F")]
    return {k: np.concatenate(v) if v else np.zeros(0) for k, v in out.items()}


@pytest.mark.parametrize("n,b", [(384, 64), (200, 64)])
def test_packed_result_is_a_tlr_operand(torch_cuda, handle, n, b):
    """tlr_pack lays the result out in the header's packed format (compared with
    the format written out in numpy), and tlr_gemm reads it back: (packed) x I
    equals the expanded result within the fp32 tolerance."""
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300.device import DeviceOperand
    rng = np.random.default_rng(21)
    A = ti.make_tlr(rng, n, b, ti.rank_uniform(0, 10), "f32")
    p = ti.Problem("times_identity", A, _identity(n, b), "N", "N", 1.0, 0.0, None, n, n, "f32")
    dc, gpu, _ = _product_then_compress(torch_cuda, handle, p, 1e-2, 16, 16)
    desc, keep = dc.pack(handle)
    torch_cuda.cuda.synchronize()
    want = _pack_numpy(gpu["tiles"], gpu["ranks"], n, b)
    bufs = keep[1]
    for k, v in want.items():
        got = bufs[k].cpu().numpy()[:v.size] if v.size else np.zeros(0)
        assert np.array_equal(got.astype(np.float64), v), k
    I = DeviceOperand(_identity(n, b))
    C = torch_cuda.full((n * n,), float("nan"), dtype=torch_cuda.float32, device="cuda")
    ws_bytes = g.tlr_gemm_workspace_bytes(handle, 0, 0, desc, I.desc, 1)
    ws = torch_cuda.empty(max(ws_bytes, 256), dtype=torch_cuda.uint8, device="cuda")
    g.tlr_gemm(handle, 0, 0, 1.0, desc, I.desc, 0.0, C.data_ptr(), n, ws.data_ptr(), ws_bytes)
    assert g.tlr_get_device_status(handle) == 0
    got = C.double().cpu().numpy().reshape(n, n).T
    ref = to.expand(gpu)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 2e-3


def test_invalid_arguments_are_refused(torch_cuda, handle):
    import gemm_tlr_gb300 as g
    from gemm_tlr_gb300 import _abi
    torch = torch_cuda
    n, b, s = 128, 64, 16
    C = torch.zeros(n * n, dtype=torch.float32, device="cuda")
    om = torch.zeros(b * s, dtype=torch.float32, device="cuda")
    U = torch.zeros(4 * b * s, dtype=torch.float32, device="cuda")
    V = torch.zeros_like(U)
    D = torch.zeros(2 * b * b, dtype=torch.float32, device="cuda")
    rk = torch.zeros(4, dtype=torch.int32, device="cuda")
    er = torch.zeros(4, dtype=torch.float32, device="cuda")
    wsb = g.tlr_compress_workspace_bytes(b, s, 4)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    host = np.zeros(n * n, dtype=np.float32)

    def call(**kw):
        a = dict(C=C.data_ptr(), ldc=n, m=n, n=n, b=b, dd=1, eps=0.1, r_max=s, om=om.data_ptr(), s=s,
                 U=U.data_ptr(), V=V.data_ptr(), D=D.data_ptr(), rk=rk.data_ptr(), er=er.data_ptr(),
                 ws=ws.data_ptr(), wsb=wsb)
        a.update(kw)
        return _abi.lib().tlr_compress(_abi._P(handle), _abi._P(a["C"]), a["ldc"], a["m"], a["n"], a["b"], a["dd"],
                                       a["eps"], a["r_max"], _abi._P(a["om"]), a["s"], _abi._P(a["U"]),
                                       _abi._P(a["V"]), _abi._P(a["D"]), _abi._P(a["rk"]), _abi._P(a["er"]),
                                       _abi._P(a["ws"]), a["wsb"])
    assert call() == 0
    assert call(s=15) == 1 and call(s=130) == 1 and call(r_max=s + 2) == 1
    assert call(ldc=n - 1) == 1 and call(eps=-1.0) == 1 and call(m=n - 1) == 1       # dense diagonal needs square
    assert call(C=host.ctypes.data) == 1                                              # host pointer
    assert call(wsb=64) == 3
    assert call(m=0, n=0) == 0
    torch.cuda.synchronize()
    assert g.tlr_get_device_status(handle) == 0


def test_large_product_sampled_tiles(torch_cuda, handle):
    """The large variable-rank product (N = 32768, b = 1024, bf16 on the tensor
    cores) with TLR output (eps = 1e-2, r_max = 96, s = 128), in the launch
    configuration of the dense product's benchmark; four tiles computed by the
    oracle one by one: a dense diagonal tile, two tiles next to the diagonal
    (their ranks above r_max: capped) and the far corner."""
    p = ti.problem(5)
    dc, gpu, _ = _product_then_compress(torch_cuda, handle, p, 1e-2, 96, 128)
    b = p.A.b
    for (i, j) in [(7, 7), (5, 6), (31, 30), (0, 31)]:
        rows, cols = np.arange(i * b, (i + 1) * b), np.arange(j * b, (j + 1) * b)
        T = oracle.gemm_problem(p, rows, cols)
        nrm = np.linalg.norm(T)
        kind, *f = gpu["tiles"][(i, j)]
        if i == j:
            assert kind == "dense" and np.linalg.norm(f[0] - T) / nrm <= 1e-2
            continue
        Uo, Vo, ro, eo = to.compress_tile(T, 1e-2, 96)
        rg, eg = int(gpu["ranks"][i, j]), float(gpu["errors"][i, j])
        e_true = np.linalg.norm(f[0] @ f[1].T - T) / nrm
        assert e_true <= np.sqrt(eg ** 2 + E2) + 1e-2, (i, j, e_true, eg)
        if ro == 96:                                     # capped on both sides
            assert rg == 96 and eo - 1e-2 <= eg <= 1.5 * eo + 1e-2, (i, j, eg, eo)
        else:
            assert eg ** 2 <= 1e-4 + E2 and ro - 2 <= rg <= 1.2 * ro + 4, (i, j, rg, ro, eg)


def test_boundary_transposed_product(torch_cuda, handle):
    """The boundary/transpose product scaled by 8 (N = 1252, b = 64: 19 full
    tiles and a 36-wide boundary, op(A) = A^T, beta = 1, fp32 on TF32 tensor
    cores) with TLR output (eps = 0.1, r_max = s = b: ranks 32-51, none capped):
    ragged boundary tiles and a dense diagonal including the corner."""
    p = ti.problem(3, scale_down=8)
    dc, gpu, _ = _product_then_compress(torch_cuda, handle, p, 0.1, 64, 64)
    ora = to.tlr_output_product(p, 0.1, 64)
    C = oracle.gemm_problem(p)
    nt = len(gpu["rdims"])
    agree = _compare_product(gpu, ora, C, 0.1, 2e-3, 64)
    assert agree >= 0.8 * nt * (nt - 1)
    assert gpu["rdims"][-1] == p.m - (nt - 1) * p.A.b          # the ragged boundary row of tiles
