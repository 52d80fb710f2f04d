"""The dense MLP block (d -> f -> d, squared-ReLU) with all six GEMMs in NVFP4 and
re-quantization between them: each stage checked against the oracle on the
GPU's own inputs to that stage (bit for bit for the activation and every
quantization, within 1e-3 for the GEMMs on identical dequantized operands)."""
import numpy as np
import pytest
import torch

from helpers import bf16_round, host_input, qtensor_to_oracle, rel_fro

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    return nv


def mlp_step(nv, X, W1, W2, dY, sr_seed=5, rht_seed=9, fused_dgrad=False, fused_fwd=False):
    """Forward and backward of one MLP block, every GEMM in NVFP4 (bf16 out).  With
    ``fused_dgrad`` (as the bench runs it) dH comes straight out of the Dgrad GEMM's
    epilogue and dA is not formed; with ``fused_fwd`` (as the bench runs it) the first
    GEMM's epilogue leaves the maxima of relu(H)^2 and its quantization skips the amax read."""
    out = {}
    out["w1q"] = nv.quantize_weight(W1)
    out["w2q"] = nv.quantize_weight(W2)
    out["xq"], out["xt"] = nv.quantize_dual(X, nv.RNE, nv.RNE, rht=True, rht_seed=rht_seed)
    maxima = None
    if fused_fwd:
        out["H"], maxima = nv.gemm_sqrelu_maxima(out["xq"], out["w1q"], rht_seed=rht_seed)
    else:
        out["H"] = nv.gemm(out["xq"], out["w1q"], torch.bfloat16)
    out["A"] = nv.sqrelu_forward(out["H"])                  # kept for the checks; the step itself
    out["aq"], out["at"] = nv.quantize_dual(out["H"], nv.RNE, nv.RNE, rht=True, rht_seed=rht_seed,
                                            pre="sqrelu", maxima=maxima)   # relu(H)^2 straight from H
    out["Y"] = nv.gemm(out["aq"], out["w2q"], torch.bfloat16)
    out["dyq"], out["dyt"] = nv.quantize_dual(dY, nv.SR, nv.SR, rht=True, sr_seed=sr_seed, sr_offset=0,
                                              rht_seed=rht_seed)
    dh_maxima = None
    if fused_dgrad:                                       # dH and its tensor maxima from the epilogue
        out["dH"], dh_maxima = nv.gemm_sqrelu_backward(out["dyq"], out["w2q"].transposed(), out["H"],
                                                       maxima=True, rht_seed=rht_seed)
    else:
        out["dA"] = nv.gemm(out["dyq"], out["w2q"].transposed(), torch.bfloat16)
        out["dH"] = nv.sqrelu_backward(out["H"], out["dA"])
    out["dW2"] = nv.gemm(out["dyt"], out["at"], torch.bfloat16)
    out["dhq"], out["dht"] = nv.quantize_dual(out["dH"], nv.SR, nv.SR, rht=True, sr_seed=sr_seed, sr_offset=1,
                                              rht_seed=rht_seed, maxima=dh_maxima)
    out["dX"] = nv.gemm(out["dhq"], out["w1q"].transposed(), torch.bfloat16)
    out["dW1"] = nv.gemm(out["dht"], out["xt"], torch.bfloat16)
    return out


def _wt(q, rows, cols):
    return dict(codes=q.codes_t.cpu().numpy(), scales=q.scales.cpu().numpy().T.copy(),
                s_dec=float(q.s_dec[0].item()), rows=rows, cols=cols, block=2)


def test_sqrelu_matches_oracle(nv, oracle_mod):
    g = torch.Generator().manual_seed(3)
    h = (torch.randn(4096, generator=g) * 3).to(torch.bfloat16)
    h[:4] = torch.tensor([0.0, -0.0, 1e-30, -1e-30])
    da = (torch.randn(4096, generator=g) * 1e-3).to(torch.bfloat16)
    hg, dag = h.cuda(), da.cuda()
    a = nv.sqrelu_forward(hg)
    dh = nv.sqrelu_backward(hg, dag)
    torch.cuda.synchronize()
    hb, db = host_input(h), host_input(da)
    assert np.array_equal(host_input(a.cpu()), oracle_mod.sqrelu_forward(hb))
    assert np.array_equal(host_input(dh.cpu()), oracle_mod.sqrelu_backward(hb, db))


def test_sqrelu_every_bf16_input_and_dense_backward(nv, oracle_mod):
    """The forward over all 65536 bf16 inputs, and the backward over every bf16 h against
    ~40 da values and every bf16 da against ~40 h values, equal the oracle (NaN results
    compared as NaN, their payload being unspecified)."""
    allb = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    a = nv.sqrelu_forward(allb.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(host_input(a.cpu()), oracle_mod.sqrelu_forward(host_input(allb)))
    rng = np.random.default_rng(17)
    part = np.concatenate([np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x3F80, 0xBF80, 0x7F7F, 0xFF7F, 0x7F80,
                                     0xFF80, 0x7FC0, 0x5F80], dtype=np.uint16),
                           rng.integers(0, 65536, 28).astype(np.uint16)])
    hb = np.concatenate([np.repeat(host_input(allb), part.size), np.tile(part, 65536)])
    db = np.concatenate([np.tile(part, 65536), np.repeat(host_input(allb), part.size)])
    to_t = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    dh = host_input(nv.sqrelu_backward(to_t(hb), to_t(db)).cpu())
    ref = oracle_mod.sqrelu_backward(hb, db)
    nan = lambda b: np.isnan(torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy())
    assert np.array_equal(nan(dh), nan(ref))
    assert np.array_equal(dh[~nan(ref)], ref[~nan(ref)])


@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused_as_benched"])
def test_mlp_block_small_full_oracle(nv, oracle_mod, fused):
    """256 tokens, 256 -> 1024 -> 256: every stage against the oracle.  ``fused`` runs the
    step the way the MLP benchmark does (relu(H)^2 quantized from the maxima the fwd1
    epilogue leaves; dH and its maxima from the dgrad2 epilogue): the quantizations of A and
    dH that skip their amax pass must still equal the oracle's quantization of the same
    tensors bit for bit, tensor scale included."""
    from nvfp4_bit_quantized_gb300 import inputs
    T, d, f = 256, 256, 1024
    X = inputs.normal((T, d), 1.0, 0, device="cuda")
    W1 = inputs.normal((f, d), 0.02, 1, device="cuda")
    W2 = inputs.normal((d, f), 0.02, 2, device="cuda")
    dY = inputs.normal((T, d), 1e-3, 3, device="cuda")
    nv.reset_status()
    o = mlp_step(nv, X, W1, W2, dY, fused_dgrad=fused, fused_fwd=fused)
    if fused:       # dA is never formed in the fused step; the plain GEMM on the same (CTA-pair)
        # kernel gives the one dH must follow bit for bit
        from nvfp4_bit_quantized_gb300 import _lib as L
        L.lib().nvfp4_gemm_force_path(2)
        try:
            o["dA"] = nv.gemm(o["dyq"], o["w2q"].transposed(), torch.bfloat16)
        finally:
            L.lib().nvfp4_gemm_force_path(0)
    assert nv.status_query() == 0
    om = oracle_mod

    def same_q(q, x_bits, block, rnd, rht=False, sr_offset=0):
        r = om.quantize(x_bits, block, rnd, rht=rht, sr_seed=5, sr_offset=sr_offset, rht_seed=9)
        assert np.array_equal(q.codes.cpu().numpy(), r["codes"])
        assert np.array_equal(q.scales.cpu().numpy(), r["scales"])
        assert np.float32(q.s_dec[0].item()) == np.float32(r["s_dec"])
        return r

    x, w1, w2, dy = host_input(X), host_input(W1), host_input(W2), host_input(dY)
    rx, rxt = same_q(o["xq"], x, om.ROW, om.RNE), same_q(o["xt"], x, om.COL, om.RNE, rht=True)
    rw1, rw2 = same_q(o["w1q"], w1, om.TILE16, om.RNE), same_q(o["w2q"], w2, om.TILE16, om.RNE)
    deq, gemm = om.dequant, om.gemm_f64
    assert rel_fro(o["H"].float().cpu().numpy(), bf16_round(gemm(deq(rx), deq(rw1)))) <= TOL
    h = host_input(o["H"])
    assert np.array_equal(host_input(o["A"]), om.sqrelu_forward(h))
    a = host_input(o["A"])
    ra, rat = same_q(o["aq"], a, om.ROW, om.RNE), same_q(o["at"], a, om.COL, om.RNE, rht=True)
    assert rel_fro(o["Y"].float().cpu().numpy(), bf16_round(gemm(deq(ra), deq(rw2)))) <= TOL
    rdy, rdyt = same_q(o["dyq"], dy, om.ROW, om.SR), same_q(o["dyt"], dy, om.COL, om.SR, rht=True)
    rw2t = om.quantize(np.ascontiguousarray(w2.T), om.TILE16)
    assert np.array_equal(o["w2q"].codes_t.cpu().numpy(), rw2t["codes"])
    assert rel_fro(o["dA"].float().cpu().numpy(), bf16_round(gemm(deq(rdy), deq(rw2t)))) <= TOL
    assert rel_fro(o["dW2"].float().cpu().numpy(), bf16_round(gemm(deq(rdyt), deq(rat)))) <= TOL
    assert np.array_equal(host_input(o["dH"]), om.sqrelu_backward(h, host_input(o["dA"])))
    dh = host_input(o["dH"])
    rdh = same_q(o["dhq"], dh, om.ROW, om.SR, sr_offset=1)
    rdht = same_q(o["dht"], dh, om.COL, om.SR, rht=True, sr_offset=1)
    rw1t = om.quantize(np.ascontiguousarray(w1.T), om.TILE16)
    assert rel_fro(o["dX"].float().cpu().numpy(), bf16_round(gemm(deq(rdh), deq(rw1t)))) <= TOL
    assert rel_fro(o["dW1"].float().cpu().numpy(), bf16_round(gemm(deq(rdht), deq(rxt)))) <= TOL


def test_mlp_block_full_size_sampled(nv, oracle_mod):
    """16384 tokens, 5120 -> 20480 -> 5120 (the MLP block workload): the activation
    bit for bit on sampled rows, each GEMM on sampled output blocks."""
    from nvfp4_bit_quantized_gb300 import inputs
    T, d, f = 16384, 5120, 20480
    X = inputs.normal((T, d), 1.0, 10, device="cuda")
    W1 = inputs.normal((f, d), 0.02, 11, device="cuda")
    W2 = inputs.normal((d, f), 0.02, 12, device="cuda")
    dY = inputs.normal((T, d), 1e-3, 13, device="cuda")
    nv.reset_status()
    o = mlp_step(nv, X, W1, W2, dY, fused_dgrad=True, fused_fwd=True)
    # dA as the separate GEMM would store it; the fused dH must equal its backward exactly
    o["dA"] = nv.gemm(o["dyq"], o["w2q"].transposed(), torch.bfloat16)
    assert torch.equal(o["dH"], nv.sqrelu_backward(o["H"], o["dA"]))
    # H and the quantization of relu(H)^2 from the epilogue's maxima equal the unfused path
    assert torch.equal(o["H"], nv.gemm(o["xq"], o["w1q"], torch.bfloat16))
    aq, at = nv.quantize_dual(o["H"], nv.RNE, nv.RNE, rht=True, rht_seed=9, pre="sqrelu")
    dhq, dht = nv.quantize_dual(o["dH"], nv.SR, nv.SR, rht=True, sr_seed=5, sr_offset=1, rht_seed=9)
    for fq, uq in ((o["aq"], aq), (o["at"], at), (o["dhq"], dhq), (o["dht"], dht)):
        assert torch.equal(fq.codes, uq.codes) and torch.equal(fq.scales, uq.scales)
        assert torch.equal(fq.s_dec[:1], uq.s_dec[:1])
    assert nv.status_query() == 0
    rng = np.random.default_rng(4)
    om = oracle_mod
    rows = [0, int(rng.integers(1, T - 1)), T - 1]
    h = o["H"][rows].cpu()
    assert np.array_equal(host_input(o["A"][rows].cpu()), om.sqrelu_forward(host_input(h)))
    assert np.array_equal(host_input(o["dH"][rows].cpu()),
                          om.sqrelu_backward(host_input(h), host_input(o["dA"][rows].cpu())))

    def check(qa, qb, D, b_tile=False, a_dict=None, b_dict=None):
        A = a_dict or qtensor_to_oracle(qa, 0)
        B = b_dict or qtensor_to_oracle(qb, 2 if b_tile else 0)
        Mr, Nr = D.shape
        Dh = D
        for m, n in ((0, 0), (Mr - 64, Nr - 64), (int(rng.integers(0, Mr // 64)) * 64, int(rng.integers(0, Nr // 64)) * 64)):
            ref = om.gemm_f64(om.dequant(A, m, m + 64), om.dequant(B, n, n + 64))
            got = Dh[m:m + 64, n:n + 64].float().cpu().numpy()
            assert rel_fro(got, bf16_round(ref)) <= TOL, (m, n)

    check(o["xq"], o["w1q"], o["H"], b_tile=True)
    check(o["aq"], o["w2q"], o["Y"], b_tile=True)
    check(o["dyq"], None, o["dA"], b_dict=_wt(o["w2q"], f, d))
    check(o["dyt"], o["at"], o["dW2"])
    check(o["dhq"], None, o["dX"], b_dict=_wt(o["w1q"], d, f))
    check(o["dht"], o["xt"], o["dW1"])


@pytest.mark.parametrize("rnd,rht", [(0, True), (1, True), (0, False)])
@pytest.mark.parametrize("shape", [(208, 336), (1024, 2048)])
def test_quantize_dual_sqrelu_equals_activation_then_quantize(nv, oracle_mod, rnd, rht, shape):
    """relu(H)^2 quantized straight from H (the activation applied as H is loaded) is bit
    for bit the quantization of the stored activation, and both equal the oracle."""
    g = torch.Generator().manual_seed(sum(shape) + rnd)
    h = (torch.randn(shape, generator=g) * 2).to(torch.bfloat16).cuda()
    h[0, :4] = torch.tensor([0.0, -0.0, -1e-30, 1e-30])
    fr, fc = nv.quantize_dual(h, rnd, rnd, rht=rht, sr_seed=3, sr_offset=1, rht_seed=5, pre="sqrelu")
    a = nv.sqrelu_forward(h)
    sr_, sc_ = nv.quantize_dual(a, rnd, rnd, rht=rht, sr_seed=3, sr_offset=1, rht_seed=5)
    torch.cuda.synchronize()
    for f, s in ((fr, sr_), (fc, sc_)):
        assert torch.equal(f.codes, s.codes) and torch.equal(f.scales, s.scales)
        assert torch.equal(f.scales_mma, s.scales_mma) and torch.equal(f.s_dec[:1], s.s_dec[:1])
    ah = oracle_mod.sqrelu_forward(host_input(h.cpu()))
    r = oracle_mod.quantize(ah, oracle_mod.ROW, rnd, sr_seed=3, sr_offset=1)
    c = oracle_mod.quantize(ah, oracle_mod.COL, rnd, rht=rht, sr_seed=3, sr_offset=1, rht_seed=5)
    assert np.array_equal(fr.codes.cpu().numpy(), r["codes"]) and np.array_equal(fc.codes.cpu().numpy(), c["codes"])
    assert np.array_equal(fr.scales.cpu().numpy(), r["scales"]) and np.array_equal(fc.scales.cpu().numpy(), c["scales"])


def _same_as_oracle(om, fr, fc, x_bits, rnd, rht, sr_seed, sr_offset, rht_seed):
    """The row and column operands quantized from epilogue maxima equal the oracle's
    quantization of the tensor: codes, canonical scales and the tensor scale."""
    r = om.quantize(x_bits, om.ROW, rnd, sr_seed=sr_seed, sr_offset=sr_offset)
    c = om.quantize(x_bits, om.COL, rnd, rht=rht, sr_seed=sr_seed, sr_offset=sr_offset, rht_seed=rht_seed)
    for q, ref in ((fr, r), (fc, c)):
        assert np.array_equal(q.codes.cpu().numpy(), ref["codes"])
        assert np.array_equal(q.scales.cpu().numpy(), ref["scales"])
        assert np.float32(q.s_dec[0].item()) == np.float32(ref["s_dec"])


@pytest.fixture
def pair_path():
    from nvfp4_bit_quantized_gb300 import _lib as L
    L.lib().nvfp4_gemm_force_path(2)
    yield
    L.lib().nvfp4_gemm_force_path(0)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (200, 296, 224), (512, 1024, 768), (384, 648, 1056),
                                   (1, 8, 32)])
def test_gemm_sqrelu_backward_equals_gemm_then_backward(nv, oracle_mod, pair_path, M, N, K):
    """The Dgrad GEMM with the squared-ReLU backward in its epilogue is bit for bit the
    CTA-pair GEMM's bf16 dA followed by the backward kernel, and that chain equals the
    oracle's backward of the GEMM output; ragged M and N, signed zeros in H."""
    g = torch.Generator().manual_seed(M + 3 * N + K)
    dy = (torch.randn((M, K), generator=g) * 1e-3).to(torch.bfloat16).cuda()
    w = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16).cuda()
    H = (torch.randn((M, N), generator=g) * 2).to(torch.bfloat16)
    H.view(-1)[:4] = torch.tensor([0.0, -0.0, 1e-30, -1e-30], dtype=torch.bfloat16)
    H = H.cuda()
    qa = nv.quantize(dy, nv.ROW, nv.SR, sr_seed=3)
    qb = nv.quantize(w, nv.ROW, nv.RNE)
    nv.reset_status()
    dH = nv.gemm_sqrelu_backward(qa, qb, H)
    dA = nv.gemm(qa, qb, torch.bfloat16)
    ref = nv.sqrelu_backward(H, dA)
    torch.cuda.synchronize()
    assert nv.status_query() == 0
    assert torch.equal(dH.view(torch.int16), ref.view(torch.int16))
    assert np.array_equal(host_input(dH.cpu()), oracle_mod.sqrelu_backward(host_input(H.cpu()), host_input(dA.cpu())))


def test_gemm_sqrelu_backward_strided(nv, pair_path):
    M, N, K = 256, 512, 512
    g = torch.Generator().manual_seed(9)
    qa = nv.quantize(torch.randn((M, K), generator=g).to(torch.bfloat16).cuda(), nv.ROW, nv.RNE)
    qb = nv.quantize((torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16).cuda(), nv.ROW, nv.RNE)
    Hbig = torch.randn((M, N + 64), generator=g).to(torch.bfloat16).cuda()
    out = torch.full((M, N + 32), 7.0, dtype=torch.bfloat16, device="cuda")
    nv.gemm_sqrelu_backward(qa, qb, Hbig[:, :N], out=out[:, :N])
    ref = nv.sqrelu_backward(Hbig[:, :N].contiguous(), nv.gemm(qa, qb, torch.bfloat16))
    torch.cuda.synchronize()
    assert torch.equal(out[:, :N], ref) and torch.all(out[:, N:] == 7.0)


@pytest.mark.parametrize("rnd,rht", [(0, True), (1, True), (0, False)])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (208, 336, 224), (512, 1024, 768), (16, 16, 32),
                                   (1040, 656, 544)])
def test_gemm_sqrelu_maxima_then_quantize_equals_unfused(nv, oracle_mod, pair_path, M, N, K, rnd, rht):
    """The first MLP GEMM with relu(H)^2's tensor maxima in its epilogue: H is bit for bit the
    CTA-pair GEMM's, and quantizing relu(H)^2 from those maxima (no amax read) gives the same
    codes, scales and tensor scales as the dual quantization with its own amax pass."""
    g = torch.Generator().manual_seed(M + 5 * N + K + rnd)
    x = torch.randn((M, K), generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn((N, K), generator=g) * 0.05).to(torch.bfloat16).cuda()
    qa, qb = nv.quantize(x, nv.ROW, nv.RNE), nv.quantize(w, nv.ROW, nv.RNE)
    nv.reset_status()
    H, m = nv.gemm_sqrelu_maxima(qa, qb, rht_seed=7)
    H2 = nv.gemm(qa, qb, torch.bfloat16)
    kw = dict(rht=rht, sr_seed=3, sr_offset=2, rht_seed=7, pre="sqrelu")
    fr, fc = nv.quantize_dual(H, rnd, rnd, maxima=m, **kw)
    ur, uc = nv.quantize_dual(H, rnd, rnd, **kw)
    torch.cuda.synchronize()
    assert nv.status_query() == 0
    assert torch.equal(H, H2)
    for f, u in ((fr, ur), (fc, uc)):
        assert torch.equal(f.codes, u.codes) and torch.equal(f.scales, u.scales)
        assert torch.equal(f.scales_mma, u.scales_mma) and torch.equal(f.s_dec[:1], u.s_dec[:1])
    # and against the oracle's quantization of relu(H)^2 itself
    a = oracle_mod.sqrelu_forward(host_input(H.cpu()))
    _same_as_oracle(oracle_mod, fr, fc, a, rnd, rht, sr_seed=3, sr_offset=2, rht_seed=7)


@pytest.mark.parametrize("rht", [True, False])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (208, 336, 224), (512, 1024, 768), (16, 16, 32)])
def test_gemm_sqrelu_backward_maxima_then_quantize_equals_unfused(nv, oracle_mod, pair_path, M, N, K, rht):
    """The fused Dgrad GEMM leaving dH's tensor maxima: dH is bit for bit the plain fused
    GEMM's, and the SR dual quantization of dH from those maxima (no amax read) equals the
    one with its own amax pass."""
    g = torch.Generator().manual_seed(2 * M + N + K)
    dy = (torch.randn((M, K), generator=g) * 1e-3).to(torch.bfloat16).cuda()
    w = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16).cuda()
    H = (torch.randn((M, N), generator=g) * 2).to(torch.bfloat16).cuda()
    qa, qb = nv.quantize(dy, nv.ROW, nv.SR, sr_seed=3), nv.quantize(w, nv.ROW, nv.RNE)
    nv.reset_status()
    dH, m = nv.gemm_sqrelu_backward(qa, qb, H, maxima=True, rht_seed=13)
    dH2 = nv.gemm_sqrelu_backward(qa, qb, H)
    kw = dict(rht=rht, sr_seed=4, sr_offset=6, rht_seed=13)
    fr, fc = nv.quantize_dual(dH, nv.SR, nv.SR, maxima=m, **kw)
    ur, uc = nv.quantize_dual(dH, nv.SR, nv.SR, **kw)
    torch.cuda.synchronize()
    assert nv.status_query() == 0
    assert torch.equal(dH.view(torch.int16), dH2.view(torch.int16))
    for f, u in ((fr, ur), (fc, uc)):
        assert torch.equal(f.codes, u.codes) and torch.equal(f.scales, u.scales)
        assert torch.equal(f.scales_mma, u.scales_mma) and torch.equal(f.s_dec[:1], u.s_dec[:1])
    # and against the oracle's quantization of dH itself
    _same_as_oracle(oracle_mod, fr, fc, host_input(dH.cpu()), nv.SR, rht, sr_seed=4, sr_offset=6, rht_seed=13)
