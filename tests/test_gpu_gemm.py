"""GEMM parity: the tcgen05 block-scaled FP4 kernel against the fp64 oracle GEMM
over the identical dequantized operands (the codes and scales the GPU wrote)."""
import numpy as np
import pytest
import torch

from helpers import bf16_round, qtensor_to_oracle, rel_fro

pytestmark = pytest.mark.gpu

TOL = 1e-3        # relative Frobenius error


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    return nv


def _operands(nv, M, N, K, seed, b_block=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = torch.randn((M, K), generator=g).to(torch.bfloat16).cuda()
    B = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16).cuda()
    qa = nv.quantize(A, nv.ROW, nv.RNE)
    qb = nv.quantize(B, b_block, nv.RNE)
    return qa, qb


def _ref(oracle_mod, qa, qb, b_block):
    return oracle_mod.gemm_f64(oracle_mod.dequant(qtensor_to_oracle(qa, 0)),
                               oracle_mod.dequant(qtensor_to_oracle(qb, b_block)))


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (384, 640, 768), (200, 300, 224), (1, 8, 32),
                                   (130, 260, 544), (256, 512, 2048)])
def test_gemm_fp32_out(nv, oracle_mod, M, N, K):
    qa, qb = _operands(nv, M, N, K, seed=M + N + K)
    nv.reset_status()
    D = nv.gemm(qa, qb, torch.float32)
    assert nv.status_query() == 0
    ref = _ref(oracle_mod, qa, qb, 0)
    err = rel_fro(D.cpu().numpy(), ref)
    assert err <= TOL, err


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (200, 300, 224)])
def test_gemm_bf16_out(nv, oracle_mod, M, N, K):
    qa, qb = _operands(nv, M, N, K, seed=7)
    D = nv.gemm(qa, qb, torch.bfloat16)
    ref = _ref(oracle_mod, qa, qb, 0)
    err = rel_fro(D.float().cpu().numpy(), bf16_round(ref))
    assert err <= TOL, err


def test_gemm_with_2d_weight_operand_and_transpose(nv, oracle_mod):
    M, N, K = 256, 512, 384
    qa, qw = _operands(nv, M, N, K, seed=11, b_block=2)
    D = nv.gemm(qa, qw, torch.float32)
    assert rel_fro(D.cpu().numpy(), _ref(oracle_mod, qa, qw, 2)) <= TOL
    # W^T as the B operand of a [*, N] x [N, K]^T product
    g = torch.Generator(device="cpu").manual_seed(12)
    dY = (torch.randn((M, N), generator=g) * 1e-3).to(torch.bfloat16).cuda()
    qd = nv.quantize(dY, nv.ROW, nv.SR, sr_seed=5)
    dX = nv.gemm(qd, qw.transposed(), torch.float32)
    wt = dict(codes=qw.codes_t.cpu().numpy(), scales=qw.scales.cpu().numpy().T.copy(),
              s_dec=float(qw.s_dec[0].item()), rows=K, cols=N, block=2)
    ref = oracle_mod.gemm_f64(oracle_mod.dequant(qtensor_to_oracle(qd, 0)), oracle_mod.dequant(wt))
    assert rel_fro(dX.cpu().numpy(), ref) <= TOL


def test_gemm_strided_output(nv, oracle_mod):
    M, N, K = 128, 256, 256
    qa, qb = _operands(nv, M, N, K, seed=13)
    big = torch.full((M, N + 40), 7.0, dtype=torch.float32, device="cuda")
    nv.gemm(qa, qb, out=big[:, :N])
    torch.cuda.synchronize()
    assert torch.all(big[:, N:] == 7.0)
    assert rel_fro(big[:, :N].cpu().numpy(), _ref(oracle_mod, qa, qb, 0)) <= TOL


def test_gemm_repeat_is_deterministic(nv):
    qa, qb = _operands(nv, 256, 512, 1024, seed=17)
    d1 = nv.gemm(qa, qb, torch.float32)
    d2 = nv.gemm(qa, qb, torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(d1, d2)


@pytest.fixture
def force_path():
    from nvfp4_bit_quantized_gb300 import _lib as L
    yield lambda path: L.lib().nvfp4_gemm_force_path(path)
    L.lib().nvfp4_gemm_force_path(0)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (512, 768, 1024), (300, 520, 352), (1000, 300, 224),
                                   (128, 256, 512), (2048, 2048, 2048)])
def test_single_cta_and_cta_pair_kernels_agree_with_oracle(nv, oracle_mod, force_path, M, N, K):
    """bf16 output through both GEMM kernels: the single-CTA tcgen05 kernel and the
    CTA-pair (cta_group::2, M = 256) kernel, ragged edges included."""
    qa, qb = _operands(nv, M, N, K, seed=M * 7 + N)
    ref = bf16_round(_ref(oracle_mod, qa, qb, 0))
    outs = {}
    for path in (1, 2):
        force_path(path)
        nv.reset_status()
        D = nv.gemm(qa, qb, torch.bfloat16)
        assert nv.status_query() == 0
        outs[path] = D.float().cpu().numpy()
        err = rel_fro(outs[path], ref)
        assert err <= TOL, (path, err)
    assert np.array_equal(outs[1], outs[2]) or rel_fro(outs[2], outs[1]) <= 1e-6


def test_operands_read_identically_by_cublaslt(nv):
    """The same codes and tensor-core scale buffers through torch._scaled_mm's block-scaled
    FP4 path (cuBLASLt), where this torch offers it: the two bf16 results differ by no more
    than two bf16 roundings, so both read the operand format the same way."""
    fp4 = getattr(torch, "float4_e2m1fn_x2", None)
    if fp4 is None:
        pytest.skip("torch has no float4_e2m1fn_x2")
    from nvfp4_bit_quantized_gb300 import inputs
    m, k, n = 1024, 2048, 768
    a = inputs.normal((m, k), 1.0, 3, device="cuda").to(torch.bfloat16)
    b = inputs.normal((n, k), 0.02, 4, device="cuda").to(torch.bfloat16)
    qa = nv.quantize(a, nv.ROW, nv.RNE)
    qb = nv.quantize(b, nv.ROW, nv.RNE)
    ours = nv.gemm(qa, qb, torch.bfloat16).float()
    try:
        lib = torch._scaled_mm(qa.codes.view(fp4), qb.codes.view(fp4).t(), qa.scales_mma.view(torch.float8_e4m3fn),
                               qb.scales_mma.view(torch.float8_e4m3fn), out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, NotImplementedError) as e:
        pytest.skip(f"block-scaled FP4 _scaled_mm not available: {e}")
    ref = lib.float() * (qa.s_dec[0] * qb.s_dec[0]).float()
    rel = ((ours - ref).norm() / ref.norm()).item()
    assert rel < 4e-3, rel


# ---- split tail (nvfp4_gemm_ws): the last partial wave's tiles cut along K over all SM pairs

def _pair_plan(M, N, K):
    """Tiles, tail tiles and parts of the split-tail schedule (one SM pair per cluster)."""
    clusters = torch.cuda.get_device_properties(0).multi_processor_count // 2
    tiles = ((M + 255) // 256) * ((N + 255) // 256)
    clusters = min(clusters, tiles)
    r = tiles % clusters
    nkt = (K + 255) // 256
    split = r != 0 and 2 * r <= clusters and nkt >= 2 and tiles // clusters < 16
    return tiles, r, (2 if split else 1)


@pytest.mark.parametrize("M,N,K", [(2048, 2560, 1024), (8192, 1280, 512), (2000, 2600, 544)])
def test_split_tail_gemm_matches_oracle_and_tile_by_tile(nv, oracle_mod, M, N, K):
    """With a workspace the tail tiles are summed from two K halves: the result stays
    within the GEMM bound of the fp64 oracle, differs from the tile-by-tile kernel only in
    those tiles (a different fp32 grouping), and is deterministic."""
    tiles, r, parts = _pair_plan(M, N, K)
    assert parts >= 2, "shape chosen to split its tail"
    qa, qb = _operands(nv, M, N, K, seed=M + 3 * N + K)
    nv.reset_status()
    d_split = nv.gemm(qa, qb, torch.bfloat16, split_tail=True)
    d_again = nv.gemm(qa, qb, torch.bfloat16, split_tail=True)
    d_whole = nv.gemm(qa, qb, torch.bfloat16)
    torch.cuda.synchronize()
    assert nv.status_query() == 0
    assert torch.equal(d_split, d_again)
    ref = bf16_round(oracle_mod.gemm_f64(oracle_mod.dequant(qtensor_to_oracle(qa, 0)),
                                         oracle_mod.dequant(qtensor_to_oracle(qb, 0)),
                                         threads=oracle_mod.host_cores()))
    assert rel_fro(d_split.float().cpu().numpy(), ref) <= TOL
    differ = (d_split != d_whole).sum().item()
    assert differ <= (r / tiles) * M * N, (differ, r, tiles)
    assert rel_fro(d_split.float().cpu().numpy(), d_whole.float().cpu().numpy()) <= 1e-3


def test_split_tail_workspace_left_ready_and_in_bounds(nv):
    """Calls of different shapes share one workspace (each leaves its counters at zero), and
    nothing is written past the declared workspace size."""
    from nvfp4_bit_quantized_gb300 import _lib as L
    nbytes = int(L.lib().nvfp4_gemm_workspace_bytes(0))
    assert nbytes > 0
    ws = torch.zeros(nbytes + 4096, dtype=torch.uint8, device="cuda")
    ws[nbytes:] = 0xA5
    import ctypes
    from nvfp4_bit_quantized_gb300.api import dev_status, _ptr, _stream

    def run(qa, qb, M, N):
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        a, b = qa.c_struct(), qb.c_struct()
        st = L.lib().nvfp4_gemm_ws(ctypes.byref(a), ctypes.byref(b), _ptr(out), L.BF16, N, _ptr(ws), nbytes,
                                   dev_status(out.device).data_ptr(), _stream())
        assert st == 0
        return out
    first = _operands(nv, 2048, 2560, 1024, seed=41)
    second = _operands(nv, 8192, 1280, 512, seed=42)
    nv.reset_status()
    o1 = run(*first, 2048, 2560)
    run(*second, 8192, 1280)
    o3 = run(*first, 2048, 2560)
    torch.cuda.synchronize()
    assert nv.status_query() == 0
    assert torch.equal(o1, o3)
    assert torch.all(ws[nbytes:] == 0xA5)
    # sum buffers and arrival counters are back at zero, ready for the next call
    assert torch.count_nonzero(ws[:nbytes]).item() == 0


def test_split_tail_gemms_on_two_streams_use_their_own_workspaces(nv):
    """Split-tail GEMMs queued on two side streams at once (no synchronisation between them) give
    the same bits as the same calls made one after another on one stream: each stream gets its own
    workspace, so their tail tiles' partial sums and counters never meet."""
    M, N, K = 2048, 2560, 1024
    assert _pair_plan(M, N, K)[2] == 2, "shape chosen to split its tail"
    qa, qb = _operands(nv, M, N, K, seed=91)
    qc, qd = _operands(nv, M, N, K, seed=92)
    nv.reset_status()
    ref1 = nv.gemm(qa, qb, torch.bfloat16, split_tail=True)
    ref2 = nv.gemm(qc, qd, torch.bfloat16, split_tail=True)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    outs1, outs2 = [], []
    for _ in range(4):
        with torch.cuda.stream(s1):
            outs1.append(nv.gemm(qa, qb, torch.bfloat16, split_tail=True))
        with torch.cuda.stream(s2):
            outs2.append(nv.gemm(qc, qd, torch.bfloat16, split_tail=True))
    torch.cuda.synchronize()
    assert nv.status_query() == 0
    for d in outs1:
        assert torch.equal(d, ref1)
    for d in outs2:
        assert torch.equal(d, ref2)
