"""GPU parity of chained products (qbw_chain_create / qbw_chain_run and
qbw_chain_run_launches): several dependent Q4_0 matrix-vector products, each
step's activations an earlier step's output, in one launch or one launch per
step.

Each step is checked against the CPU oracle applied to the step's actual
input, the chain's own bf16 output of the earlier step read back after the
run, with the matvec bound (2e-3 of sum |w x| plus the bf16 output rounding)
or the gate+up bound.  On the decode sweep's shapes every step must also equal
the separate qmv_q4_0 / qmv_gateup_q4_0 call on the same input bit for bit:
both run the same 8-bit tensor-core arithmetic over the same unit split.
"""
import numpy as np
import pytest

import synth
from tolerance import check_gateup, check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev(a_bits):
    return torch.from_numpy(a_bits.view(np.int16).copy()).view(torch.bfloat16).cuda()


def bits(t):
    """bf16 device tensor -> uint16 bit patterns (the oracle's bf16 input form)."""
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def check_step(oracle, w, w_up, x_bits, y, N, K, what):
    out_bf16 = y.dtype == torch.bfloat16
    if w_up is None:
        y_ref, S = oracle.qmv("q4_0", w, x_bits, N, K)
        return check_matvec(to_f64(y), y_ref, S, out_bf16=out_bf16, what=what)
    ref = oracle.gateup_q4_0(w, w_up, x_bits, N, K)
    check_gateup(to_f64(y), ref, oracle, out_bf16=out_bf16, what=what)
    return 0.0


def test_chain_small_mixed_steps(qbw, oracle):
    # x0 -> s0 (1024 x 512) -> s1 gate+up (512 x 1024) -> s2 (700 x 512, a
    # ragged tile) ; s3 reads an earlier step's output (y0[:768]), fp32 out.
    x0 = synth.activations(512, seed=71, dtype="bf16")
    shapes = [(1024, 512, False), (512, 1024, True), (700, 512, False), (256, 768, False)]
    ws = []
    for i, (N, K, gu) in enumerate(shapes):
        wg = synth.q4_0_weights(N, K, seed=72 + i, stream=0)
        wu = synth.q4_0_weights(N, K, seed=72 + i, stream=1) if gu else None
        ws.append((wg, wu))
    xd = bf16_dev(x0)
    y0 = torch.empty(1024, dtype=torch.bfloat16, device="cuda")
    y1 = torch.empty(512, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty(700, dtype=torch.bfloat16, device="cuda")
    y3 = torch.full((256,), float("nan"), dtype=torch.float32, device="cuda")
    dw = [(dev_u8(a), None if b is None else dev_u8(b)) for a, b in ws]
    steps = [(dw[0][0], None, xd, y0, 1024, 512), (dw[1][0], dw[1][1], y0, y1, 512, 1024),
             (dw[2][0], None, y1, y2, 700, 512), (dw[3][0], None, y0[:768], y3, 256, 768)]
    chain = qbw.Chain(steps)
    try:
        for rep in range(2):           # a second run must find the counter and scratch reset
            chain.run()
            torch.cuda.synchronize()
            assert qbw.fault_read(clear=True) == 0
            ins = [x0, bits(y0), bits(y1), bits(y0)[:768]]
            outs = [y0, y1, y2, y3]
            for i, ((N, K, gu), (wg, wu)) in enumerate(zip(shapes, ws)):
                check_step(oracle, wg, wu, ins[i], outs[i], N, K, f"chain step {i} run {rep}")
    finally:
        chain.close()


def test_chain_single_step_matches_bound(qbw, oracle):
    N, K = 3000, 2048
    w = synth.q4_0_weights(N, K, seed=80)
    x = synth.activations(K, seed=80, dtype="bf16")
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    chain = qbw.Chain([(dev_u8(w), None, bf16_dev(x), y, N, K)])
    try:
        chain.run()
        torch.cuda.synchronize()
        assert qbw.fault_read(clear=True) == 0
        worst = check_step(oracle, w, None, x, y, N, K, "chain single step")
        assert worst < 1e-3
    finally:
        chain.close()


HIDDEN, QDIM, KVDIM, FFN = 5376, 8192, 4096, 21504


@pytest.mark.parametrize("mode", ["one_launch", "launches"])
def test_chain_decode_layers_match_separate_calls(qbw, oracle, mode):
    # two layers of the decode sweep: h -> q|k|v -> o(q) -> gate+up(o) -> down -> h;
    # run as one cooperative launch, or as one launch per step that prefetches
    # the next step's first weight tiles into L2 (qbw_chain_run_launches)
    layers = 2
    W = []
    for layer in range(layers):
        W.append({"qkv": dev_u8(synth.q4_0_weights(QDIM + 2 * KVDIM, HIDDEN, seed=90, stream=0, layer=layer)),
                  "o": dev_u8(synth.q4_0_weights(HIDDEN, QDIM, seed=90, stream=1, layer=layer)),
                  "g": dev_u8(synth.q4_0_weights(FFN, HIDDEN, seed=90, stream=2, layer=layer)),
                  "u": dev_u8(synth.q4_0_weights(FFN, HIDDEN, seed=90, stream=3, layer=layer)),
                  "d": dev_u8(synth.q4_0_weights(HIDDEN, FFN, seed=90, stream=4, layer=layer))})
    h0 = synth.activations(HIDDEN, seed=91, dtype="bf16")
    bf = torch.bfloat16
    hs = [bf16_dev(h0)] + [torch.empty(HIDDEN, dtype=bf, device="cuda") for _ in range(layers)]
    qkv = [torch.empty(QDIM + 2 * KVDIM, dtype=bf, device="cuda") for _ in range(layers)]
    o = [torch.empty(HIDDEN, dtype=bf, device="cuda") for _ in range(layers)]
    a = [torch.empty(FFN, dtype=bf, device="cuda") for _ in range(layers)]
    steps = []
    for L in range(layers):
        steps += [(W[L]["qkv"], None, hs[L], qkv[L], QDIM + 2 * KVDIM, HIDDEN),
                  (W[L]["o"], None, qkv[L][:QDIM], o[L], HIDDEN, QDIM),
                  (W[L]["g"], W[L]["u"], o[L], a[L], FFN, HIDDEN),
                  (W[L]["d"], None, a[L], hs[L + 1], HIDDEN, FFN)]
    chain = qbw.Chain(steps)
    try:
        if mode == "launches":
            chain.run_launches()
        else:
            chain.run()
        torch.cuda.synchronize()
        assert qbw.fault_read(clear=True) == 0
        # each step against the separate call on the chain's own input, bit for bit
        for i, (w, w_up, x, y, N, K) in enumerate(steps):
            ref = torch.empty_like(y)
            if w_up is None:
                qbw.qmv_q4_0(w, x, ref, 1, N, K)
            else:
                qbw.qmv_gateup_q4_0(w, w_up, x, ref, 1, N, K)
            torch.cuda.synchronize()
            assert torch.equal(ref.view(torch.int16), y.view(torch.int16)), f"step {i}: chain != separate call"
        # and the first layer's steps against the oracle
        L0 = [("qkv", None, bits(hs[0]), qkv[0], QDIM + 2 * KVDIM, HIDDEN),
              ("o", None, bits(qkv[0])[:QDIM], o[0], HIDDEN, QDIM),
              ("g", "u", bits(o[0]), a[0], FFN, HIDDEN),
              ("d", None, bits(a[0]), hs[1], HIDDEN, FFN)]
        host = {k: v.cpu().numpy() for k, v in W[0].items()}
        for name, up, xb, y, N, K in L0:
            check_step(oracle, host[name], None if up is None else host[up], xb, y, N, K, f"layer 0 {name}")
    finally:
        chain.close()


def test_chain_rejects_bad_steps(qbw):
    N, K = 256, 512
    w = torch.zeros(N * K // 32 * 18, dtype=torch.uint8, device="cuda")
    x = torch.zeros(K, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qbw.QbwError, match="QBW_ESHAPE"):
        qbw.Chain([(w, None, x, y, N, 300)])                      # K % 256 != 0
    with pytest.raises(qbw.QbwError, match="QBW_EALIGN"):
        xs = torch.zeros(K + 8, dtype=torch.bfloat16, device="cuda")
        qbw.Chain([(w, None, xs[1:], y, N, K)])                   # x off 16 bytes
    with pytest.raises(qbw.QbwError, match="QBW_EINVAL"):
        xy = torch.zeros(K, dtype=torch.bfloat16, device="cuda")
        qbw.Chain([(w, None, xy, xy[:N], N, K)])                  # y overlaps its x
    with pytest.raises(qbw.QbwError, match="QBW_EINVAL"):
        wy = torch.zeros(N * K // 32 * 18, dtype=torch.uint8, device="cuda")
        qbw.Chain([(wy, None, x, y, N, K), (w, None, y, wy.view(torch.bfloat16)[:N], N, K)])   # y over weights
    with pytest.raises(qbw.QbwError, match="QBW_EDTYPE"):
        qbw.Chain([(w, None, x, torch.zeros(N, dtype=torch.float16, device="cuda"), N, K)])


def test_chain_one_group_steps_and_fp32_gateup(qbw, oracle):
    # K = 256: one K-group per tile, so every unit is a whole tile; the last
    # step is a gate+up with fp32 output
    x0 = synth.activations(256, seed=95, dtype="bf16")
    w0 = synth.q4_0_weights(256, 256, seed=96)
    wg = synth.q4_0_weights(300, 256, seed=97, stream=0)
    wu = synth.q4_0_weights(300, 256, seed=97, stream=1)
    y0 = torch.empty(256, dtype=torch.bfloat16, device="cuda")
    y1 = torch.empty(300, dtype=torch.float32, device="cuda")
    chain = qbw.Chain([(dev_u8(w0), None, bf16_dev(x0), y0, 256, 256),
                       (dev_u8(wg), dev_u8(wu), y0, y1, 300, 256)])
    try:
        chain.run()
        torch.cuda.synchronize()
        assert qbw.fault_read(clear=True) == 0
        check_step(oracle, w0, None, x0, y0, 256, 256, "chain K=256 step 0")
        check_step(oracle, wg, wu, bits(y0), y1, 300, 256, "chain K=256 gate+up")
    finally:
        chain.close()
