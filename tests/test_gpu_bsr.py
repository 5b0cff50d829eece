"""BSR SpMM on the tensor cores (bf16 in, fp32 accumulate) against the fp64
oracle: exact small-integer cases, identity blocks, empty and long block-rows
(ring wrap-around), several column tiles, padded leading dimensions, and the
16384^2 64x64-block workload at N = 1024 on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from csr_bsr_spmv_gb300 import spx
from gpu_util import BF16_ABS, BF16_REL, assert_within

pytestmark = pytest.mark.gpu


def bits_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def run_bsr(M, K, brp, bcol, bval_bits, B_bits, N, ldb=None, ldc=None):
    ldb = ldb or N
    ldc = ldc or N
    Bfull = np.zeros((K, ldb), np.uint16)
    Bfull[:, :N] = B_bits
    Bd = bits_dev(Bfull)[:, :N]
    Cd = torch.full((M, ldc), -7.0, device="cuda")
    spx.spx_spmm_bsr(M, K, 64, 64, torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                     bits_dev(bval_bits.reshape(-1)), Bd, Cd[:, :N])
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    out = Cd.cpu().numpy()
    assert np.all(out[:, N:] == -7.0)
    return out[:, :N]


def pattern(seed, MB, KB, counts):
    """Block pattern with the given number of blocks per block-row."""
    cols = []
    for I, c in enumerate(counts):
        cols.append(np.sort(synth.permutation(seed * 1000 + I, KB)[:c]).astype(np.int32))
    brp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return brp, np.concatenate(cols).astype(np.int32) if cols else np.zeros(0, np.int32)


def test_small_integers_exact():
    """Entries and B in {-3..3}: every product and partial sum is an exact
    integer in fp32, so the result equals the dense product exactly."""
    MB, KB, N = 4, 8, 128
    brp, bcol = pattern(1, MB, KB, [3, 0, 8, 1])
    nb = bcol.size
    A = np.floor(synth.uniform(1, synth.T_VAL, nb * 4096, -3, 4)).astype(np.float32).reshape(nb, 64, 64)
    B = np.floor(synth.uniform(1, synth.T_B, KB * 64 * N, -3, 4)).astype(np.float32).reshape(KB * 64, N)
    got = run_bsr(MB * 64, KB * 64, brp, bcol, synth.to_bf16_bits(A), synth.to_bf16_bits(B).reshape(B.shape), N)
    dense = np.zeros((MB * 64, KB * 64))
    for I in range(MB):
        for b in range(brp[I], brp[I + 1]):
            dense[I * 64:(I + 1) * 64, bcol[b] * 64:(bcol[b] + 1) * 64] = A[b]
    assert np.array_equal(got, dense @ B.astype(np.float64))


def test_identity_blocks():
    """Block-diagonal identity: C = B exactly (checks the MN-major / K-major
    operand layouts and the TMEM lane -> output mapping)."""
    MB, N = 6, 256
    brp = np.arange(MB + 1, dtype=np.int32)
    bcol = np.arange(MB, dtype=np.int32)
    eye = np.tile(np.eye(64, dtype=np.float32), (MB, 1, 1))
    B = synth.uniform(2, synth.T_B, MB * 64 * N).reshape(MB * 64, N)
    Bb = synth.to_bf16_bits(B).reshape(B.shape)
    got = run_bsr(MB * 64, MB * 64, brp, bcol, synth.to_bf16_bits(eye), Bb, N)
    assert np.array_equal(got, synth.bf16_bits_to_f32(Bb))


def test_permutation_blocks():
    """One permutation block per block-row (shifted block columns): rows of B
    land permuted, exactly."""
    MB, KB, N = 3, 5, 128
    perm = synth.permutation(3, 64)
    P = np.eye(64, dtype=np.float32)[perm]
    brp = np.arange(MB + 1, dtype=np.int32)
    bcol = np.array([4, 0, 2], np.int32)
    B = synth.uniform(3, synth.T_B, KB * 64 * N).reshape(KB * 64, N)
    Bb = synth.to_bf16_bits(B).reshape(B.shape)
    got = run_bsr(MB * 64, KB * 64, brp, bcol, synth.to_bf16_bits(np.stack([P] * MB)), Bb, N)
    Bf = synth.bf16_bits_to_f32(Bb).reshape(B.shape)
    for I in range(MB):
        assert np.array_equal(got[I * 64:(I + 1) * 64], Bf[bcol[I] * 64:(bcol[I] + 1) * 64][perm])


@pytest.mark.parametrize("counts,N,ldb,ldc", [
    ([1, 2, 3, 4], 128, None, None),
    ([0, 5, 0, 9, 17], 256, None, None),        # empty block-rows, ring wrap-around
    ([33, 1], 384, 512, 400),                    # padded leading dimensions
    ([7] * 12, 640, None, None),
])
def test_random_blocks(counts, N, ldb, ldc):
    MB, KB = len(counts), 40
    brp, bcol = pattern(4, MB, KB, counts)
    nb = bcol.size
    A = synth.normal_bf16(4, synth.T_VAL, nb * 4096, 0.02).reshape(nb, 64, 64)
    B = synth.normal_bf16(4, synth.T_B, KB * 64 * N, 1.0).reshape(KB * 64, N)
    got = run_bsr(MB * 64, KB * 64, brp, bcol, A, B, N, ldb, ldc)
    ref, bound = oracle.bsr_spmm(MB * 64, KB * 64, 64, 64, brp, bcol, A, B)
    assert_within(got, ref, bound, BF16_REL, BF16_ABS, what=f"counts={counts}")
    # fp32 accumulation is in fact far tighter than the bf16 bound
    assert_within(got, ref, bound, 1e-5, 1e-6, what="fp32-level")


def test_bad_arguments_rejected_without_launch():
    lib = spx._lib()
    before = spx.launch_count()
    z = torch.zeros(64 * 1024, dtype=torch.int32, device="cuda")
    p = spx._ptr(z)
    assert lib.spx_spmm_bsr(64, 64, 0, 32, 1, p, p, p, 128, p, 128, 1.0, 0.0, p, 128, None) == -1    # br <= 0
    assert lib.spx_spmm_bsr(64, 64, 64, 64, 1, p, p, p, 128, p, 100, 1.0, 0.0, p, 128, None) == -1   # ldb < N
    assert lib.spx_spmm_bsr(64, 64, 64, 64, 1, p, p, p, 128, p, 132, 1.0, 0.0, p, 128, None) == -8   # ldb % 8 (64 x 64)
    assert lib.spx_spmm_bsr(64, 64, 16, 8, 1, p, p, p, 128, p, 131, 1.0, 0.0, p, 128, None) == -8    # odd ldb (others)
    assert lib.spx_spmm_bsr(64, 64, 16, 8, 1, p, p, p + 2, 128, p + 2, 130, 1.0, 0.0, p, 128, None) == -8  # B 2-byte
    assert lib.spx_spmm_bsr(64, 64, 16, 16, 1 << 27, p, p, p, 128, p, 128, 1.0, 0.0, p, 128, None) == -2  # nnzb*bc
    # the block-row split is built for 64-row block-rows only
    plan = spx.BsrPlan(64, 0, torch.zeros(2, dtype=torch.int32))
    assert lib.spx_spmm_bsr_planned(plan.handle, 64, 64, 16, 16, 0, p, p, p, 128, p, 128, 1.0, 0.0, p, 128, None, 0,
                                    None) == -7
    assert spx.launch_count() == before


def _bsr_case(seed, M, K, br, bc, lmin, lmax, values="uniform"):
    d = synth.random_coo(seed, M, K, lmin, lmax, values)
    vb = synth.to_bf16_bits(d["val"])
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], vb)
    brp, bcol, bval, _ = oracle.build_bsr(M, K, rp, col, val, br, bc)
    return brp, bcol, bval


def _gamma(n, u=2.0 ** -24):
    return n * u / (1 - n * u)


def _tc_shape(br, bc):
    """Shapes the tensor-core kernel takes (with ldb a multiple of 8 and 16-byte aligned arrays)."""
    return (br, bc) == (64, 64) or (br % 16 == 0 and 16 <= br <= 128 and bc % 16 == 0 and (bc <= 64 or bc % 64 == 0))


SHAPES = [
    (37, 29, 1, 1, 64),
    (100, 90, 2, 2, 130),
    (97, 203, 3, 5, 77),
    (256, 256, 4, 4, 512),
    (300, 260, 8, 8, 129),
    (512, 384, 16, 16, 256),
    (200, 330, 32, 32, 96),
    (190, 400, 16, 64, 200),
    (400, 190, 64, 16, 200),
    (333, 333, 64, 32, 65),
    (300, 500, 128, 128, 130),
    (250, 250, 100, 70, 33),
    (64, 70, 1, 64, 8),
    (70, 64, 64, 1, 1),
    (230, 700, 48, 48, 300),
    (260, 520, 32, 128, 136),
    (330, 400, 112, 64, 129),
    (290, 600, 96, 192, 64),
    (100, 300, 128, 16, 257),
]


@pytest.mark.parametrize("M,K,br,bc,N", SHAPES)
@pytest.mark.parametrize("beta", [0.0, 0.5])
@pytest.mark.parametrize("layout", ["cuda-core", "tensor-core"])
def test_general_block_shapes(M, K, br, bc, N, beta, layout):
    """Block shapes other than 64 x 64: ragged M, K, N, padded leading
    dimensions, alpha/beta; against the oracle within the fp32 accumulation
    bound of each element's term count, nothing written outside the M x N part
    of C, and beta = 0 never reading C (NaN there stays out).  With ldb a
    multiple of 8, shapes whose sides are multiples of 16 (bc <= 64 or a
    multiple of 64, br <= 128) run on the tensor cores; with an ldb that is
    not, and for every other shape, on the CUDA cores."""
    if layout == "tensor-core" and not _tc_shape(br, bc):
        pytest.skip("not a tensor-core shape")
    brp, bcol, bval = _bsr_case(11 + br * 7 + bc, M, K, br, bc, 0, 40)
    B = synth.normal_bf16(12, synth.T_B, K * N, 1.0).reshape(K, N)
    C0 = synth.uniform(13, synth.T_Y, M * N).reshape(M, N).astype(np.float32)
    if layout == "tensor-core":
        ldb, ldc = (N + 7) // 8 * 8 + 8, N + 3
    else:
        ldb, ldc = N + (N % 2) + 6, N + 3
        if ldb % 8 == 0:
            ldb += 2
    Bfull = np.zeros((K, ldb), np.uint16)
    Bfull[:, :N] = B
    Bd = bits_dev(Bfull)[:, :N]
    Cfull = torch.full((M + 1, ldc), -7.0, device="cuda")
    Cd = Cfull[:M, :N]
    Cd.copy_(torch.from_numpy(C0) if beta != 0.0 else torch.full((M, N), float("nan")))
    spx.spx_spmm_bsr(M, K, br, bc, torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                     bits_dev(bval.reshape(-1)), Bd, Cd, alpha=1.5, beta=beta)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    out = Cfull.cpu().numpy()
    assert np.all(out[:M, N:] == -7.0) and np.all(out[M] == -7.0)
    got = out[:M, :N]
    ref, bound = oracle.bsr_spmm(M, K, br, bc, brp, bcol, bval, B, alpha=1.5, beta=beta,
                                 C=C0 if beta != 0.0 else None)
    nterm = int(np.diff(brp).max(initial=0)) * bc
    # the tensor cores' fp32 accumulation is not specified to round to nearest: bound it with a unit
    # roundoff of 2^-23 (any faithful rounding) there, 2^-24 for the CUDA cores' fused multiply-adds
    rel = _gamma(nterm + 3, 2.0 ** -23 if layout == "tensor-core" else 2.0 ** -24)
    assert_within(got, ref, bound, rel, 0.0, what=f"{br}x{bc} {layout}")
    # bitwise the same on a second call
    Cd2 = torch.from_numpy(C0).cuda() if beta != 0.0 else torch.zeros(M, N, device="cuda")
    spx.spx_spmm_bsr(M, K, br, bc, torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                     bits_dev(bval.reshape(-1)), Bd, Cd2, alpha=1.5, beta=beta)
    assert np.array_equal(Cd2.cpu().numpy().view(np.uint32), got.view(np.uint32))


@pytest.mark.parametrize("br,bc,N", [(4, 4, 70), (16, 8, 70), (3, 7, 70), (96, 48, 70), (16, 16, 72), (32, 64, 72),
                                     (128, 128, 136), (48, 192, 64)])
def test_general_shapes_small_integers_exact(br, bc, N):
    """Entries and B small integers: every product and partial sum is exact in
    fp32, so the result equals the dense product exactly (N = 70: the CUDA
    cores; N a multiple of 8 with 16-multiple sides: the tensor cores)."""
    M, K = 180, 150
    brp, bcol, bval = _bsr_case(21 + br, M, K, br, bc, 0, 30, "int")
    B = np.floor(synth.uniform(22, synth.T_B, K * N, -3, 4)).astype(np.float32).reshape(K, N)
    Bb = synth.to_bf16_bits(B).reshape(K, N)
    Cd = torch.full((M, N), -7.0, device="cuda")
    spx.spx_spmm_bsr(M, K, br, bc, torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                     bits_dev(bval.reshape(-1)), bits_dev(Bb), Cd)
    torch.cuda.synchronize()
    dense = np.zeros(((M + br - 1) // br * br, (K + bc - 1) // bc * bc))
    Af = synth.bf16_bits_to_f32(bval.reshape(-1)).reshape(bval.shape)
    for I in range(brp.size - 1):
        for b in range(brp[I], brp[I + 1]):
            dense[I * br:(I + 1) * br, bcol[b] * bc:(bcol[b] + 1) * bc] = Af[b]
    assert np.array_equal(Cd.cpu().numpy(), dense[:M, :K] @ B.astype(np.float64))


def test_general_shape_empty_and_long_block_rows():
    """Empty block-rows (C = beta C) next to a block-row of every block column
    (chunk boundaries inside a block, many chunks)."""
    M, K, br, bc, N = 5 * 12, 40 * 12, 12, 12, 96
    counts = [0, 40, 3, 0, 17]
    brp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    bcol = np.concatenate([np.sort(synth.permutation(31 + I, 40)[:c]) for I, c in enumerate(counts)]).astype(np.int32)
    nb = bcol.size
    A = synth.normal_bf16(31, synth.T_VAL, nb * br * bc, 0.5).reshape(nb, br, bc)
    B = synth.normal_bf16(32, synth.T_B, K * N, 1.0).reshape(K, N)
    C0 = synth.uniform(33, synth.T_Y, M * N).reshape(M, N).astype(np.float32)
    Cd = torch.from_numpy(C0.copy()).cuda()
    spx.spx_spmm_bsr(M, K, br, bc, torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                     bits_dev(A.reshape(-1)), bits_dev(B), Cd, alpha=-1.0, beta=2.0)
    torch.cuda.synchronize()
    ref, bound = oracle.bsr_spmm(M, K, br, bc, brp, bcol, A, B, alpha=-1.0, beta=2.0, C=C0)
    assert_within(Cd.cpu().numpy(), ref, bound, _gamma(40 * bc + 3), 0.0, what="empty/long")
    got = Cd.cpu().numpy()
    assert np.array_equal(got[:br], (2.0 * C0[:br]).astype(np.float32))


@pytest.mark.parametrize("alpha,beta", [(2.0, 0.0), (-0.5, 1.5), (1.0, -1.0)])
def test_alpha_beta(alpha, beta):
    MB, KB, N = 5, 12, 256
    brp, bcol = pattern(6, MB, KB, [4, 0, 7, 2, 11])
    nb = bcol.size
    A = synth.normal_bf16(6, synth.T_VAL, nb * 4096, 0.02).reshape(nb, 64, 64)
    B = synth.normal_bf16(6, synth.T_B, KB * 64 * N, 1.0).reshape(KB * 64, N)
    C0 = synth.uniform(6, synth.T_Y, MB * 64 * N).reshape(MB * 64, N)
    Cd = torch.from_numpy(C0.copy()).cuda()
    spx.spx_spmm_bsr(MB * 64, KB * 64, 64, 64, torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                     bits_dev(A.reshape(-1)), bits_dev(B), Cd, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    ref, bound = oracle.bsr_spmm(MB * 64, KB * 64, 64, 64, brp, bcol, A, B, alpha=alpha, beta=beta, C=C0)
    assert_within(Cd.cpu().numpy(), ref, bound, BF16_REL, BF16_ABS, what=f"alpha={alpha} beta={beta}")


def test_no_blocks_gives_zero():
    M, K, N = 128, 128, 128
    brp = np.zeros(3, np.int32)
    got = run_bsr(M, K, brp, np.zeros(0, np.int32), np.zeros((0, 64, 64), np.uint16),
                  np.ones((K, N), np.uint16), N)
    assert not got.any()


def test_no_blocks_scales_by_beta():
    M, K, N = 128, 64, 256
    C0 = synth.uniform(9, synth.T_Y, M * N).reshape(M, N)
    Cd = torch.from_numpy(C0.copy()).cuda()
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    spx.spx_spmm_bsr(M, K, 64, 64, torch.zeros(3, dtype=torch.int32, device="cuda"), z[:0], z[:0].to(torch.int16),
                     torch.zeros(K, N, dtype=torch.int16, device="cuda"), Cd, beta=-2.0)
    torch.cuda.synchronize()
    assert np.array_equal(Cd.cpu().numpy(), np.float32(-2.0) * C0)


@pytest.mark.slow
def test_block_sparse_full_size_sampled():
    """16384^2 with 64x64 blocks, 26 per block-row (nnzb = 6656), B 16384 x 1024:
    two sampled rows of every block-row, built through the library's
    COO -> CSR -> BSR path."""
    cfg = synth.block_sparse()
    M, K, N = cfg["M"], cfg["K"], cfg["N"]
    rp, col, val = spx.spx_build_csr(M, K, cfg["row"], cfg["col"], cfg["val_bf16"])
    brp, bcol, bval, fill = spx.spx_build_bsr(M, K, rp, col, val, 64, 64)
    assert bcol.size == 6656 and fill == 1.0
    Cd = torch.empty(M, N, device="cuda")
    spx.spx_spmm_bsr(M, K, 64, 64, torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                     bits_dev(bval.reshape(-1)), bits_dev(cfg["B_bf16"]), Cd)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    rng = np.random.default_rng(5)
    rows = np.sort(np.concatenate([np.arange(0, M, 64) + rng.integers(0, 64, M // 64),
                                   np.arange(0, M, 64) + 63])).astype(np.int32)
    got = Cd[torch.from_numpy(rows).long().cuda()].cpu().numpy()
    ref, bound = oracle.bsr_spmm(M, K, 64, 64, brp, bcol, bval, cfg["B_bf16"], rows=rows)
    assert_within(got, ref, bound, BF16_REL, BF16_ABS, what="block-sparse full size")


def _skewed_bsr(M, N, seed=9):
    c = synth.block_sparse_skewed(seed, M=M, N=N)
    rp, col, val = oracle.build_csr(M, c["K"], c["row"], c["col"], c["val_bf16"])
    brp, bcol, bval, _ = oracle.build_bsr(M, c["K"], rp, col, val, 64, 64)
    dev_args = (torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                torch.from_numpy(np.ascontiguousarray(bval).reshape(-1).view(np.int16)).cuda())
    return c, rp, col, val, brp, dev_args


@pytest.mark.parametrize("max_blocks", [0, 1, 8, 27])
@pytest.mark.parametrize("N,alpha,beta", [(128, 1.0, 0.0), (256, -0.5, 1.5)])
def test_planned_task_split(max_blocks, N, alpha, beta):
    """Long block-rows split into pieces (partial tiles + fixed-order fix-up) against the
    fp64 oracle; reproducible; the plain call meets the same bound."""
    M = 2048
    c, rp, col, val, brp, (dbrp, dbcol, dbval) = _skewed_bsr(M, N)
    K = c["K"]
    P = spx.BsrPlan(M, dbcol.numel(), dbrp, max_chunks=max_blocks)
    assert max_blocks == 0 or P.info["split_windows"] > 0
    dB = torch.from_numpy(c["B_bf16"].view(np.int16)).cuda()
    C0 = synth.uniform(N, synth.T_Y, M * N).reshape(M, N)
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(val), synth.bf16_bits_to_f32(c["B_bf16"]), alpha, beta,
                             C0)
    outs = []
    for _ in range(2):
        Cd = torch.from_numpy(C0.copy()).cuda()
        spx.spx_spmm_bsr_planned(P, M, K, 64, 64, dbrp, dbcol, dbval, dB, Cd, alpha, beta)
        torch.cuda.synchronize()
        assert spx.spx_last_device_error() == 0
        outs.append(Cd)
    assert_within(outs[0].cpu().numpy(), ref, bound, rel=BF16_REL, ab=BF16_ABS, what=f"planned bsr max={max_blocks}")
    assert torch.equal(outs[0], outs[1])
    C3 = torch.from_numpy(C0.copy()).cuda()
    spx.spx_spmm_bsr(M, K, 64, 64, dbrp, dbcol, dbval, dB, C3, alpha=alpha, beta=beta)
    if P.info["split_windows"] == 0:
        # no task split: the same products; the plain call may still cut its last round of tiles in two
        # (head and tail pieces added in another order), so the two agree to fp32 rounding
        assert_within(C3.cpu().numpy(), outs[0].cpu().numpy().astype(np.float64), bound, what="plain vs planned")
    assert_within(C3.cpu().numpy(), ref, bound, rel=BF16_REL, ab=BF16_ABS, what="plain bsr")


def test_planned_errors():
    M, N = 1024, 128
    c, rp, col, val, brp, (dbrp, dbcol, dbval) = _skewed_bsr(M, N)
    K = c["K"]
    dB, C = torch.from_numpy(c["B_bf16"].view(np.int16)).cuda(), torch.empty(M, N, device="cuda")
    P = spx.BsrPlan(M, dbcol.numel(), brp, max_chunks=4)
    cases = [(lambda: spx.spx_spmm_bsr_planned(spx.BsrPlan(M, dbcol.numel(), brp, max_chunks=4, upload=False), M, K,
                                               64, 64, dbrp, dbcol, dbval, dB, C), -10),
             (lambda: spx.spx_spmm_bsr_planned(P, M, K, 64, 64, dbrp, dbcol, dbval, dB, C,
                                               scratch=torch.zeros(4, device="cuda")), -1),
             (lambda: spx.spx_spmm_bsr_planned(P, M - 64, K, 64, 64, dbrp, dbcol, dbval, dB, C[:M - 64]), -1)]
    for f, code in cases:
        with pytest.raises(spx.SpxError) as e:
            f()
        assert e.value.code == code


@pytest.mark.slow
def test_planned_skewed_full_size_sampled():
    """16,384^2 with every 16th block-row 8x longer (208 blocks), N = 1024, default split; two rows per block-row."""
    M, N = 16384, 1024
    c, rp, col, val, brp, (dbrp, dbcol, dbval) = _skewed_bsr(M, N)
    K = c["K"]
    P = spx.BsrPlan(M, dbcol.numel(), brp)
    assert P.info["split_windows"] == M // 64 // 16
    Cd = torch.empty(M, N, device="cuda")
    spx.spx_spmm_bsr_planned(P, M, K, 64, 64, dbrp, dbcol, dbval, torch.from_numpy(c["B_bf16"].view(np.int16)).cuda(),
                             Cd)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    rows = np.sort(np.concatenate([np.arange(0, M, 64), np.arange(41, M, 64)])).astype(np.int32)
    ref, bound = oracle.spmm(M, rp, col, synth.bf16_bits_to_f32(val), synth.bf16_bits_to_f32(c["B_bf16"]), rows=rows)
    got = Cd[torch.from_numpy(rows).long().cuda()].cpu().numpy()
    assert_within(got, ref, bound, rel=BF16_REL, ab=BF16_ABS, what="planned bsr skewed full size")


def _ragged_bsr(M, K, seed, lmax=40):
    """A random CSR (bf16 values) and its BSR with 64 x 64 blocks; M and K need not be multiples of 64."""
    d = synth.random_coo(seed, M, K, 1, lmax)
    vb = synth.to_bf16_bits(d["val"])
    rp, col, val = oracle.build_csr(M, K, d["row"], d["col"], vb)
    brp, bcol, bval, _ = oracle.build_bsr(M, K, rp, col, val, 64, 64)
    return brp, bcol, np.ascontiguousarray(bval)


@pytest.mark.parametrize("M,K,N", [(100, 130, 200), (64 * 3 + 1, 128, 8), (64, 63, 40), (1, 1, 1000),
                                   (300, 500, 129), (257, 700, 384)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, -1.5)])
@pytest.mark.parametrize("split", [False, True])
def test_ragged_shapes(M, K, N, alpha, beta, split):
    """Any M, K, N: a ragged last block-row / block column (zero-padded in the BSR arrays, B rows past K
    read as zeros) and a ragged last 128-column tile; nothing is written outside the M x N part of C.
    split: the planned call with block-rows cut into pieces of two blocks."""
    brp, bcol, bval = _ragged_bsr(M, K, 90 + M + N)
    ldb, ldc = (N + 7) // 8 * 8 + 8, N + 3
    Bb = synth.to_bf16_bits(synth.uniform(91, synth.T_B, K * N)).reshape(K, N)
    Bfull = np.zeros((K, ldb), np.uint16)
    Bfull[:, :N] = Bb
    C0 = synth.uniform(92, synth.T_Y, M * ldc).reshape(M, ldc)
    Cd = torch.from_numpy(C0.copy()).cuda()
    dbrp, dbcol, dbval = torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(), bits_dev(bval.reshape(-1))
    dB = bits_dev(Bfull)[:, :N]
    if split:
        P = spx.BsrPlan(M, bcol.size, dbrp, max_chunks=2)
        spx.spx_spmm_bsr_planned(P, M, K, 64, 64, dbrp, dbcol, dbval, dB, Cd[:, :N], alpha, beta)
    else:
        spx.spx_spmm_bsr(M, K, 64, 64, dbrp, dbcol, dbval, dB, Cd[:, :N], alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    assert spx.spx_last_device_error() == 0
    got = Cd.cpu().numpy()
    assert np.array_equal(got[:, N:], C0[:, N:])  # columns past N untouched
    ref, bound = oracle.bsr_spmm(M, K, 64, 64, brp, bcol, bval, Bb, alpha=alpha, beta=beta, C=C0[:, :N])
    assert_within(got[:, :N], ref, bound, BF16_REL, BF16_ABS, what=f"M={M} K={K} N={N} split={split}")


def test_bounded_wait_runs_out_and_reports_timeout():
    """A wait that nothing completes gives up after its limit (about 1 ms here), the device error word
    then reads SPX_ERR_TIMEOUT exactly once, and the context stays usable: a BSR product right after is
    exact."""
    assert spx.spx_last_device_error() == 0
    spx.spx_wait_probe(2_000_000)
    assert spx.spx_last_device_error() == -6
    assert spx.spx_last_device_error() == 0
    test_small_integers_exact()
    assert spx.spx_last_device_error() == 0


@pytest.mark.parametrize("MB,KB,per_row,N,beta", [(20, 80, 60, 256, 0.0), (20, 80, 60, 200, 0.5),
                                                  (64, 70, 64, 1024, -1.0), (9, 40, 31, 384, 0.0)])
def test_last_round_cut_in_two(MB, KB, per_row, N, beta):
    """When the last round of tiles leaves at least half the resident CTAs idle and block-rows hold 48 blocks or
    more on average, its tiles are cut in two: a head piece stored by the first launch, a tail piece added by a
    second launch (two launches).  Against the oracle (bf16 bound and fp32 rounding), with beta, reproducibly,
    with nothing written past column N; a pattern below the 48-block average stays whole (one launch)."""
    counts = [per_row] * MB
    brp, bcol = pattern(7, MB, KB, counts)
    nb = bcol.size
    A = synth.normal_bf16(7, synth.T_VAL, nb * 4096, 0.02).reshape(nb, 64, 64)
    B = synth.normal_bf16(7, synth.T_B, KB * 64 * N, 1.0).reshape(KB * 64, N)
    C0 = synth.uniform(7, synth.T_Y, MB * 64 * N).reshape(MB * 64, N)
    ntiles = MB * ((N + 127) // 128)
    G = 3 * torch.cuda.get_device_properties(0).multi_processor_count  # the persistent kernel's resident CTAs
    R = ntiles % G
    cut = R > 0 and 2 * R <= G and per_row >= 48
    outs = []
    for _ in range(2):
        Cd = torch.from_numpy(C0.copy()).cuda()
        before = spx.launch_count()
        spx.spx_spmm_bsr(MB * 64, KB * 64, 64, 64, torch.from_numpy(brp).cuda(), torch.from_numpy(bcol).cuda(),
                         bits_dev(A.reshape(-1)), bits_dev(B), Cd, alpha=1.0, beta=beta)
        torch.cuda.synchronize()
        assert spx.launch_count() - before == (2 if cut else 1)
        assert spx.spx_last_device_error() == 0
        outs.append(Cd.cpu().numpy())
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    ref, bound = oracle.bsr_spmm(MB * 64, KB * 64, 64, 64, brp, bcol, A, B, alpha=1.0, beta=beta, C=C0)
    assert_within(outs[0], ref, bound, BF16_REL, BF16_ABS, what=f"cut={cut}")
    assert_within(outs[0], ref, bound, 1e-5, 1e-6, what="fp32-level")
