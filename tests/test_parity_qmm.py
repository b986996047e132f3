"""GPU parity of the small-M tensor-core product qmm_q4_0_smallM (prefill
tiles of up to 32 tokens) against the CPU oracle on the same seeded bytes.

The pass rule is 1e-2 of S = sum_k |x w| per output (weights are rounded to
bf16 once on chip: at most 2^-8 relative; the bf16 activations are exact),
plus half an ulp of bf16 when the output is bf16.  Every output is compared,
small shapes and the full-size ones (5376 x 5376 and 5376 x 21504, M = 8, 16,
32) alike.
"""
import numpy as np
import pytest

import synth
from tolerance import check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).cuda()


def workspace(qbw, M, N, K):
    nbytes = qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K)
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda"), nbytes


def run_qmm(qbw, w, X, M, N, K, odt, calls=2):
    # several calls on one workspace: its counters must come back to zero
    ws, nbytes = workspace(qbw, M, N, K)
    wd, Xd = dev_u8(w), dev_bf16(X)
    outs = []
    for _ in range(calls):
        Y = torch.full((M, N), float("nan"), dtype=odt, device="cuda")
        qbw.qmm_q4_0_smallM(wd, Xd, Y, M, N, K, workspace=ws)
        outs.append(Y)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    for Y in outs[1:]:
        assert torch.equal(Y.view(torch.int16) if odt == torch.bfloat16 else Y.view(torch.int32),
                           outs[0].view(torch.int16) if odt == torch.bfloat16 else outs[0].view(torch.int32))
    return to_f64(outs[0])


@pytest.mark.parametrize("M", [1, 3, 8, 16, 17, 32])
@pytest.mark.parametrize("N,K", [(128, 256), (300, 512), (1000, 2304), (129, 4096), (64, 96)])
@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float32])
def test_qmm_small(qbw, oracle, M, N, K, odt):
    w = synth.q4_0_weights(N, K, seed=N + K + M)
    X = synth.activations((M, K), seed=M * 31 + K, dtype="bf16")
    Y = run_qmm(qbw, w, X, M, N, K, odt)
    Y_ref, S = oracle.qmm_q4_0(w, X, M, N, K)
    check_matvec(Y, Y_ref, S, rel=1e-2, out_bf16=(odt == torch.bfloat16), what=f"qmm M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [8, 16, 32])
@pytest.mark.parametrize("K", [5376, 21504])
def test_qmm_full_size(qbw, oracle, M, K):
    # the small-M tile workload in full: every row of every token
    N = 5376
    w = synth.q4_0_weights(N, K, seed=3)
    X = synth.activations((M, K), seed=3, dtype="bf16")
    Y = run_qmm(qbw, w, X, M, N, K, torch.bfloat16)
    Y_ref, S = oracle.qmm_q4_0(w, X, M, N, K)
    check_matvec(Y, Y_ref, S, rel=1e-2, out_bf16=True, what=f"qmm full M={M} K={K}")


# (M, N, K, whether a 152-SM GB300 runs the K-splits of a tile as one cluster).
# Splits per tile = min(152 // tiles, K / 256); one CTA per SM holds clusters
# of 2, 3, 4, 5, 6 and 7 CTAs 76, 46, 36, 28, 23 and 15 at a time, so 20 tiles
# of 7 splits do not all fit and take the workspace path.
CLUSTER_CASES = [(8, 4352, 2048, True), (32, 3328, 2048, True), (5, 2816, 1536, True), (16, 300, 512, True),
                 (32, 8192, 1024, True), (8, 2560, 2048, False)]


@pytest.mark.parametrize("M,N,K,cluster", CLUSTER_CASES)
def test_qmm_cluster_split_shapes(qbw, oracle, M, N, K, cluster):
    # 2 .. 8 K-splits per 128-row tile: the splits of a tile add their partial
    # sums in distributed shared memory, with no workspace, when all the
    # tiles' clusters fit on the device at once
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert (qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K) == 0) == cluster
    w = synth.q4_0_weights(N, K, seed=N + M)
    X = synth.activations((M, K), seed=M + 7, dtype="bf16")
    Y_ref, S = oracle.qmm_q4_0(w, X, M, N, K)
    for odt in (torch.float32, torch.bfloat16):
        Y = run_qmm(qbw, w, X, M, N, K, odt, calls=3)
        check_matvec(Y, Y_ref, S, rel=1e-2, out_bf16=(odt == torch.bfloat16), what=f"qmm cluster M={M} N={N} K={K}")


# Stream-K shapes (M <= 16): whole-tile splits would leave SMs idle, so one CTA
# per SM takes an equal range of (tile, K-group) units; ranges cross tile
# boundaries and the tiles are finished from the other CTAs' published shares.
# (M, N, K): 42 tiles x 84 groups (ranges of 23..24 units, 3..4 CTAs per
# tile); 32 tiles with a 32-row tail; 3 and 4 tokens (column padding); 60
# tiles x 64 groups.
STREAMK_CASES = [(8, 5376, 21504), (16, 4000, 21504), (3, 5376, 21504), (4, 4000, 21504), (13, 7680, 16384)]


@pytest.mark.parametrize("M,N,K", STREAMK_CASES)
def test_qmm_streamk_shapes(qbw, oracle, M, N, K):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        # the shares' layout: a 4096-byte counter region, then [152][M rounded
        # up to 4][128] 64-bit words
        mp = (M + 3) // 4 * 4
        assert qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K) == 4096 + (152 * mp * 128 * 8 + 255) // 256 * 256
    w = synth.q4_0_weights(N, K, seed=N + 3 * M)
    X = synth.activations((M, K), seed=M + 29, dtype="bf16")
    Y_ref, S = oracle.qmm_q4_0(w, X, M, N, K)
    for odt in (torch.float32, torch.bfloat16):
        Y = run_qmm(qbw, w, X, M, N, K, odt, calls=3)
        check_matvec(Y, Y_ref, S, rel=1e-2, out_bf16=(odt == torch.bfloat16), what=f"qmm stream-K M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(16384, 5376), (5413, 5376), (600, 65536)])
@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float32])
def test_qmm_one_two_tokens_exact_path(qbw, oracle, M, N, K, odt):
    # M <= 2 with at least 15 MB of weights runs on the exact-code M = 1
    # kernel (the two tokens take the x_hi / x_lo columns): it needs no
    # workspace and meets the M = 1 bound, 2e-3 of sum |w x|
    assert qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K) == 0
    w = synth.q4_0_weights(N, K, seed=N + M)
    X = synth.activations((M, K), seed=M + 17, dtype="bf16")
    Y = run_qmm(qbw, w, X, M, N, K, odt, calls=2)
    Y_ref, S = oracle.qmm_q4_0(w, X, M, N, K)
    check_matvec(Y, Y_ref, S, rel=2e-3, out_bf16=(odt == torch.bfloat16), what=f"qmm exact M={M} N={N} K={K}")


def test_qmm_deterministic(qbw):
    M, N, K = 32, 1024, 5376
    w = dev_u8(synth.q4_0_weights(N, K, seed=9))
    X = dev_bf16(synth.activations((M, K), seed=9, dtype="bf16"))
    ws, _ = workspace(qbw, M, N, K)
    Y1 = torch.empty(M, N, device="cuda")
    Y2 = torch.empty(M, N, device="cuda")
    qbw.qmm_q4_0_smallM(w, X, Y1, M, N, K, workspace=ws)
    qbw.qmm_q4_0_smallM(w, X, Y2, M, N, K, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int32), Y2.view(torch.int32))


def test_qmm_constant_weights_closed_form(qbw, oracle):
    # every weight d * (c - 8) with d = 0.5, c = 11: Y[m, n] = 1.5 * sum_k X[m, k]
    M, N, K = 8, 256, 2048
    w = synth.constant_blocks("q4_0", N, K, 0x3800, 11)
    X = synth.activations((M, K), seed=2, dtype="bf16")
    Y = run_qmm(qbw, w, X, M, N, K, torch.float32)
    Y_ref, S = oracle.qmm_q4_0(w, X, M, N, K)
    check_matvec(Y, Y_ref, S, rel=1e-2, what="constant")
    zero = synth.constant_blocks("q4_0", N, K, 0x3C00, 8)
    Yz = run_qmm(qbw, zero, X, M, N, K, torch.float32)
    assert np.all(Yz == 0.0)


def test_qmm_workspace_too_small_is_rejected(qbw):
    # 5 tiles of 128 rows, 16 K-splits each: more splits than one cluster takes
    M, N, K = 16, 640, 4096
    need = qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K)
    if need == 0:
        pytest.skip("this device plans no split for the shape")
    w = dev_u8(synth.q4_0_weights(N, K, seed=1))
    X = dev_bf16(synth.activations((M, K), seed=1, dtype="bf16"))
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    small = torch.zeros(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(qbw.QbwError) as e:
        qbw.qmm_q4_0_smallM(w, X, Y, M, N, K, workspace=small)
    assert e.value.status == 6


def test_qmm_workspace_shared_across_shapes(qbw):
    # One workspace, zero-filled once, serves calls of different shapes in turn:
    # every call must find its arrival counters at zero and, for a stream-K
    # plan, its share words untagged, whatever an earlier shape left behind
    # (the last shape is a stream-K plan, run after workspace-path ones).
    shapes = [(16, 5376, 5376), (17, 256, 2048), (32, 128, 21504), (8, 640, 4096), (32, 1024, 5376),
              (8, 4000, 21504)]
    size = max(qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K) for M, N, K in shapes)
    if size == 0:
        pytest.skip("this device plans no split for these shapes")
    shared = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for i, (M, N, K) in enumerate(shapes):
        w = dev_u8(synth.q4_0_weights(N, K, seed=40 + i))
        X = dev_bf16(synth.activations((M, K), seed=40 + i, dtype="bf16"))
        fresh, _ = workspace(qbw, M, N, K)
        Y_fresh = torch.empty(M, N, device="cuda")
        Y_shared = torch.empty(M, N, device="cuda")
        qbw.qmm_q4_0_smallM(w, X, Y_fresh, M, N, K, workspace=fresh)
        qbw.qmm_q4_0_smallM(w, X, Y_shared, M, N, K, workspace=shared)
        torch.cuda.synchronize()
        assert torch.equal(Y_shared.view(torch.int32), Y_fresh.view(torch.int32)), (M, N, K)
    assert qbw.fault_read(clear=True) == 0


@pytest.mark.parametrize("M,N,K", [(32, 2048, 256), (8, 4096, 512)])
def test_qmm_weight_rounded_once(qbw, oracle, M, N, K):
    # Token m is the unit vector e_k(m), so Y[m, n] is the tile's bf16 weight
    # W[n, k(m)] itself (one product with 1, fp32 sums of zeros).  Rounded once
    # from the exact (c - 8) d it is within 2^-8 (1 + 2^-7) of it, relative; a
    # scale rounded to bf16 before the product would put a quarter of the
    # weights beyond that.
    w = synth.q4_0_weights(N, K, seed=M + N)
    ks = (np.arange(M) * 37 + 5) % K
    X = np.zeros((M, K), dtype=np.uint16)
    X[np.arange(M), ks] = 0x3F80                      # bf16 1.0
    Y = run_qmm(qbw, w, X, M, N, K, torch.float32)
    W = oracle.dequant("q4_0", w, N, K).astype(np.float64)   # exact (c - 8) d
    ref = W[:, ks].T                                  # [M, N]
    err = np.abs(Y - ref)
    assert np.all(err <= 2.0 ** -8 * (1 + 2.0 ** -7) * np.abs(ref)), \
        f"max relative error {np.max(err / np.maximum(np.abs(ref), 1e-300)):.3e}"
    # and each value is a bf16 number
    assert np.all((Y.astype(np.float32).view(np.uint32) & 0xFFFF) == 0)
