"""Unit tests of the library's GEMM kernels through the muon_debug_gemm hook,
against PyTorch fp32 products of the same operands.  Ordered from the
smallest single-tile case up, so a layout or descriptor slip shows up in the
simplest shape that exhibits it."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    import newton_schulz_04_gb300 as m
    m.load(build_if_missing=True)
    return m


def _rel(a, b):
    return (a - b).norm().item() / max(b.norm().item(), 1e-30)


def _ref(A, B, b_mn):
    A = A.float()
    B = B.float()
    return A @ B if b_mn else A @ B.transpose(1, 2)


def _rand(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype).cuda()


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (256, 256, 256), (256, 512, 384), (512, 768, 1024)])
def test_tc_gemm_kmajor_b(M, N, K):
    m = _lib()
    A = _rand((2, M, K), 1)
    B = _rand((2, N, K), 2)
    out = m.debug_gemm(A, B)
    torch.cuda.synchronize()
    # same bf16 operands, fp32 accumulation on both sides: only summation order
    # and the 16-bit output pair (2^-17 relative per element) differ
    assert _rel(out, _ref(A, B, False)) < 2e-5


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (256, 512, 256), (512, 1024, 512)])
def test_tc_gemm_mnmajor_b(M, N, K):
    m = _lib()
    A = _rand((2, M, K), 3)
    B = _rand((2, K, N), 4)
    out = m.debug_gemm(A, B, b_mn=True)
    torch.cuda.synchronize()
    assert _rel(out, _ref(A, B, True)) < 2e-5


def block_lower(S, device="cuda"):
    """Mask of the 256 x 256 blocks on or below the diagonal (symmetric storage)."""
    r = torch.arange(S, device=device) // 256
    return r[:, None] >= r[None, :]


@pytest.mark.parametrize("S,K", [(256, 128), (512, 256), (768, 1024)])
def test_tc_syrk_block_lower(S, K):
    m = _lib()
    X = _rand((3, S, K), 5)
    out = m.debug_gemm(X, X, sym=True)
    torch.cuda.synchronize()
    ref = _ref(X, X, False)
    mask = block_lower(S)
    assert _rel(out[:, mask], ref[:, mask]) < 2e-5


@pytest.mark.parametrize("split", [1, 3])
def test_tc_symmetric_operands_in_block_lower_storage(split):
    # Upper blocks of both operands hold NaN: the kernel must never read them
    # (it reads the transposed lower block instead) and still form P G exactly.
    m = _lib()
    g = torch.Generator().manual_seed(17)
    S = 768
    X = torch.randn(2, S, S, generator=g, dtype=torch.float64)
    Gs = (X @ X.transpose(1, 2)) / S
    Ps = Gs @ Gs - 0.5 * Gs
    mask = block_lower(S, "cpu")
    def store(x):
        h, l = _split(x.float().cuda())
        h[:, ~mask.cuda()] = float("nan")
        l[:, ~mask.cuda()] = float("nan")
        return h, l
    Ph, Pl = store(Ps)
    Gh, Gl = store(Gs)
    if split == 1:
        out = m.debug_gemm(Ph, Gh, sym=True, a_sym=True, b_sym=True)
        full = lambda t: torch.where(mask.cuda(), t, t.transpose(1, 2))  # noqa: E731
        ref = _ref(full(Ph.float()), full(Gh.float()), False)
        tol = 2e-5
    else:
        out = m.debug_gemm(Ph, Gh, Pl, Gl, split=3, sym=True, a_sym=True, b_sym=True)
        ref = (Ps @ Gs).float().cuda()
        tol = 4e-5
    torch.cuda.synchronize()
    mk = mask.cuda()
    assert torch.isfinite(out[:, mk]).all()
    assert _rel(out[:, mk], ref[:, mk]) < tol


def test_tc_rect_with_symmetric_a_operand():
    # B X with B symmetric in block-lower storage (the original-space update)
    m = _lib()
    g = torch.Generator().manual_seed(18)
    S, L = 512, 768
    Y = torch.randn(S, S, generator=g, dtype=torch.float64)
    Bs = ((Y + Y.T) / 2).float().cuda()[None]
    X = torch.randn(1, S, L, generator=g).to(torch.bfloat16).cuda()
    Bh = Bs.to(torch.bfloat16)
    mask = block_lower(S)
    Bst = Bh.clone()
    Bst[:, ~mask] = float("nan")
    out = m.debug_gemm(Bst, X, b_mn=True, a_sym=True)
    torch.cuda.synchronize()
    assert _rel(out, _ref(Bh, X, True)) < 2e-5


def _split(x32):
    hi = x32.to(torch.bfloat16)
    lo = (x32 - hi.float()).to(torch.bfloat16)
    return hi, lo


@pytest.mark.parametrize("b_mn", [False, True])
def test_tc_gemm_split3(b_mn):
    m = _lib()
    g = torch.Generator().manual_seed(6)
    A32 = torch.randn(2, 256, 512, generator=g).cuda()
    B32 = (torch.randn(2, 512, 512, generator=g) if b_mn else torch.randn(2, 512, 512, generator=g)).cuda()
    Ah, Al = _split(A32)
    Bh, Bl = _split(B32)
    out = m.debug_gemm(Ah, Bh, Al, Bl, split=3, b_mn=b_mn)
    torch.cuda.synchronize()
    ref = _ref(A32.double(), B32.double(), b_mn).float()
    one = _ref(Ah, Bh, b_mn)
    # three products of ~8-bit operands reach ~16-bit operand accuracy
    assert _rel(out, ref) < 4e-5
    assert _rel(one, ref) > 1e-3


def test_tc_gemm_split2_mnmajor():
    m = _lib()
    g = torch.Generator().manual_seed(12)
    A32 = torch.randn(2, 256, 512, generator=g).cuda()
    B = torch.randn(2, 512, 768, generator=g).to(torch.bfloat16).cuda()
    Ah, Al = _split(A32)
    out = m.debug_gemm(Ah, B, Al, None, split=2, b_mn=True)
    torch.cuda.synchronize()
    ref = (A32.double() @ B.double()).float()
    assert _rel(out, ref) < 4e-5
    assert _rel(_ref(Ah, B, True), ref) > 1e-3


def test_tc_sym_split3_symmetric_operands():
    m = _lib()
    g = torch.Generator().manual_seed(7)
    X = torch.randn(2, 512, 512, generator=g, dtype=torch.float64)
    Gs = (X @ X.transpose(1, 2)) / 512
    Ps = Gs @ Gs - 0.5 * Gs
    Gh, Gl = _split(Gs.float().cuda())
    Ph, Pl = _split(Ps.float().cuda())
    out = m.debug_gemm(Ph, Gh, Pl, Gl, split=3, sym=True)
    torch.cuda.synchronize()
    ref = (Ps @ Gs).float().cuda()
    mask = block_lower(512)
    assert _rel(out[:, mask], ref[:, mask]) < 4e-5


# ---- fp16 operands (the original-space schedule's steps after the first)

@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (512, 768, 1024)])
def test_tc_gemm_fp16_operands(M, N, K, b_mn):
    m = _lib()
    A = _rand((2, M, K), 31, torch.float16)
    B = _rand((2, K, N) if b_mn else (2, N, K), 32, torch.float16)
    out = m.debug_gemm(A, B, b_mn=b_mn)
    torch.cuda.synchronize()
    ref = _ref(A.double(), B.double(), b_mn).float()
    # exact fp16 operands, fp32 accumulation, a ~22-bit fp16 output pair
    assert _rel(out, ref) < 2e-5
    # the same bits read as bf16 would give a different product: the type is honoured
    wrong = _ref(A.view(torch.bfloat16).double(), B.view(torch.bfloat16).double(), b_mn).float()
    assert _rel(wrong, ref) > 0.5


def test_tc_fp16_output_pair_residual_is_scaled():
    # out + lo / 2^11 reconstructs the fp32 accumulator to ~22 bits; the head
    # alone is only fp16-accurate
    m = _lib()
    A = _rand((1, 256, 256), 33, torch.float16)
    B = _rand((1, 256, 256), 34, torch.float16)
    ref = _ref(A.double(), B.double(), False).float()
    lib = m.load()
    import ctypes
    out = torch.zeros(1, 256, 256, dtype=torch.float16, device="cuda")
    lo = torch.zeros_like(out)
    ws = m.new_workspace(4096)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.muon_debug_gemm(p(A), None, p(B), None, 1, 256, 256, 256, 1, 0, 0, 2, p(out), p(lo), p(ws),
                             ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    head = _rel(out.float(), ref)
    full = _rel(out.float() + lo.float() / 2048.0, ref)
    assert 1e-4 < head < 1e-3        # fp16 rounding, 2^-12 relative on average
    assert full < 2e-6
    # the stored residual is scaled up, so it sits well above fp16's subnormals
    assert lo.abs().max().item() > 2 ** -14


def test_tc_fp16_symmetric_operands_in_block_lower_storage():
    m = _lib()
    g = torch.Generator().manual_seed(35)
    S = 768
    X = torch.randn(2, S, S, generator=g, dtype=torch.float64)
    Gs = (X @ X.transpose(1, 2)) / S
    mask = block_lower(S, "cpu")
    Gh = Gs.to(torch.float16).cuda()
    Gst = Gh.clone()
    Gst[:, ~mask.cuda()] = float("nan")
    out = m.debug_gemm(Gst, Gst, sym=True, a_sym=True, b_sym=True)
    torch.cuda.synchronize()
    ref = _ref(Gh.double(), Gh.double(), False).float()
    mk = mask.cuda()
    assert torch.isfinite(out[:, mk]).all()
    assert _rel(out[:, mk], ref[:, mk]) < 2e-5


# ---- scaled fp16 pairs (split 5): the low parts stored as (v - hi) * 2^11

def _f16_pair(x64):
    hi = x64.to(torch.float16)
    lo = ((x64 - hi.double()) * 2048.0).to(torch.float16)
    return hi, lo


@pytest.mark.parametrize("M,N,K,b_mn", [(256, 256, 128, False), (256, 512, 384, True), (512, 768, 1024, False),
                                        (768, 256, 512, True)])
def test_tc_fp16_pair_products(M, N, K, b_mn):
    """C = (A + A_lo/2^11)(B + B_lo/2^11) to about 22 bits: the two low-part
    products accumulate at 2^11 times their scale, and the tensor core scales
    that accumulator by 2^-11 before the high-part product adds to it."""
    m = _lib()
    g = torch.Generator().manual_seed(40 + M + K)
    A64 = torch.randn(2, M, K, generator=g, dtype=torch.float64)
    B64 = torch.randn(2, K, N, generator=g, dtype=torch.float64) if b_mn else \
        torch.randn(2, N, K, generator=g, dtype=torch.float64)
    Ah, Al = _f16_pair(A64)
    Bh, Bl = _f16_pair(B64)
    out = m.debug_gemm(Ah.cuda(), Bh.cuda(), A_lo=Al.cuda(), B_lo=Bl.cuda(), split=5, b_mn=b_mn)
    torch.cuda.synchronize()
    Ap = Ah.double() + Al.double() / 2048.0
    Bp = Bh.double() + Bl.double() / 2048.0
    ref = (Ap @ Bp if b_mn else Ap @ Bp.transpose(1, 2)).float()
    out = out.cpu()
    # about 22-bit operands; the tensor cores' fp32 accumulation (about 1e-6 of
    # the sum of |products|) sets the bound
    assert _rel(out, ref) < 5e-6
    # the high parts alone are 2^-11-accurate, so the low-part terms are really in
    hh = (Ah.double() @ Bh.double() if b_mn else Ah.double() @ Bh.double().transpose(1, 2)).float()
    assert _rel(hh, ref) > 1e-4


def test_tc_fp16_pair_symmetric_operands_in_block_lower_storage():
    """Split 5 on symmetric operands given block-lower (the upper k-blocks of
    both parts read as transposed boxes), with a symmetric output."""
    m = _lib()
    g = torch.Generator().manual_seed(47)
    S = 768
    X = torch.randn(1, S, S, generator=g, dtype=torch.float64)
    G64 = (X @ X.transpose(1, 2)) / S
    Gh, Gl = _f16_pair(G64)
    mask = block_lower(S, "cpu")
    Ghs, Gls = Gh.clone(), Gl.clone()
    Ghs[:, ~mask] = float("nan")
    Gls[:, ~mask] = float("nan")
    out = m.debug_gemm(Ghs.cuda(), Ghs.cuda(), A_lo=Gls.cuda(), B_lo=Gls.cuda(), split=5, sym=True, a_sym=True,
                       b_sym=True).cpu()
    torch.cuda.synchronize()
    Gp = Gh.double() + Gl.double() / 2048.0
    ref = (Gp @ Gp).float()
    assert torch.isfinite(out[:, mask]).all()
    assert _rel(out[:, mask], ref[:, mask]) < 5e-6


def test_tc_fp16_pair_rejects_bf16_and_missing_parts():
    m = _lib()
    A = _rand((1, 256, 128), 48, torch.float16)
    B = _rand((1, 256, 128), 49, torch.float16)
    with pytest.raises(m.MuonError):
        m.debug_gemm(A, B, A_lo=A, split=5)  # no B_lo
    with pytest.raises(m.MuonError):
        m.debug_gemm(A.to(torch.bfloat16), B.to(torch.bfloat16), A_lo=A.to(torch.bfloat16),
                     B_lo=B.to(torch.bfloat16), split=5)


# ---- diagonal K segment: C = A B + B_lo / 2^11 with the second term on the tensor cores

@pytest.mark.parametrize("M,N,batch,a_sym", [(256, 256, 1, False), (512, 768, 2, False), (1024, 256, 3, True),
                                             (768, 512, 2, True)])
def test_tc_diagonal_segment(M, N, batch, a_sym):
    m = _lib()
    g = torch.Generator().manual_seed(36 + M + N)
    if a_sym:
        X = torch.randn(batch, M, M, generator=g, dtype=torch.float64)
        A64 = (X + X.transpose(1, 2)) / (2 * M)
    else:
        A64 = torch.randn(batch, M, M, generator=g, dtype=torch.float64) / M
    A = A64.to(torch.float16)
    B = torch.randn(batch, M, N, generator=g).to(torch.float16)
    B_lo = torch.randn(batch, M, N, generator=g).to(torch.float16)
    Ad = A.clone()
    if a_sym:  # block-lower storage: the upper blocks must never be read
        Ad[:, ~block_lower(M, "cpu")] = float("nan")
    out = m.debug_gemm(Ad.cuda(), B.cuda(), B_lo=B_lo.cuda(), split=4, b_mn=True, a_sym=a_sym)
    torch.cuda.synchronize()
    prod = A.double() @ B.double()
    ref = prod + B_lo.double() / 2048.0
    out = out.cpu()
    assert torch.isfinite(out).all()
    # every row block gets its own rows of B_lo (a row offset error is O(1) relative)
    assert _rel(out, ref.float()) < 2e-5
    assert _rel(prod.float(), ref.float()) > 1e-3  # the segment's term is well above the tolerance


def test_tc_diagonal_segment_rejects_unsupported_forms():
    m = _lib()
    A = _rand((1, 256, 256), 37, torch.float16)
    B = _rand((1, 256, 512), 38, torch.float16)
    with pytest.raises(m.MuonError):  # needs B's residual
        m.debug_gemm(A, B, split=4, b_mn=True)
    with pytest.raises(m.MuonError):  # K-major B
        m.debug_gemm(A, B.transpose(1, 2).contiguous(), B_lo=B, split=4, b_mn=False)
    with pytest.raises(m.MuonError):  # bf16 operands
        m.debug_gemm(A.view(torch.bfloat16), B.view(torch.bfloat16), B_lo=B.view(torch.bfloat16), split=4,
                     b_mn=True)
    A2 = _rand((1, 256, 512), 39, torch.float16)  # K != M
    B2 = _rand((1, 512, 256), 40, torch.float16)
    with pytest.raises(m.MuonError):
        m.debug_gemm(A2, B2, B_lo=B2, split=4, b_mn=True)


@pytest.mark.parametrize("M,N,K,b_mn,sym", [(128, 128, 16, False, False), (256, 384, 80, True, False),
                                             (384, 384, 48, False, True)])
def test_simt_gemm(M, N, K, b_mn, sym):
    m = _lib()
    A = _rand((2, M, K), 8, torch.float32)
    B = _rand((2, K, N) if b_mn else (2, N, K), 9, torch.float32)
    if sym:
        B = A
    out = m.debug_gemm(A, B, b_mn=b_mn, sym=sym)
    torch.cuda.synchronize()
    ref = _ref(A.double(), B.double(), b_mn).float()
    assert _rel(out, ref) < 1e-6


def test_bounded_wait_reports_timeout_and_context_survives():
    m = _lib()
    ws = m.new_workspace(4096)
    m.debug_bounded_wait(ws, 2_000_000)  # ~1 ms of SM cycles, nobody arrives
    assert m.device_status(ws) == 6  # MUON_ERR_TIMEOUT
    assert m.device_status(ws) == 0  # cleared
    A = _rand((1, 256, 128), 10)
    B = _rand((1, 256, 128), 11)
    out = m.debug_gemm(A, B, workspace=ws)
    torch.cuda.synchronize()
    assert _rel(out, _ref(A, B, False)) < 2e-5
    assert m.device_status(ws) == 0


def test_tc_accumulation_precision():
    """Characterises the fp32 accumulation of the tensor-core kernel: exact bf16
    operands, a 256x256 output (one CTA pair), K from 256 to 16384, against the fp64 product
    (printed with -s; the bounds hold with margin on GB300)."""
    m = _lib()
    g = torch.Generator().manual_seed(0)
    print("\n| K | rel_fro | rel_vs_q | max err / sum abs | cuBLAS fp32 rel |")
    for K, bound in [(256, 1e-5), (1024, 1e-5), (4096, 2e-5), (16384, 6e-5)]:
        A = torch.randn(1, 256, K, generator=g).to(torch.bfloat16)
        B = torch.randn(1, 256, K, generator=g).to(torch.bfloat16)
        ref = A.double() @ B.double().transpose(1, 2)
        out = m.debug_gemm(A.cuda(), B.cuda()).cpu().double()
        r32 = ref.float()
        h = r32.to(torch.bfloat16).float()
        refq = (h + (r32 - h).to(torch.bfloat16).float()).double()
        rel_fro = ((out - ref).norm() / ref.norm()).item()
        rel_q = ((out - refq).norm() / ref.norm()).item()
        sumabs = A.double().abs() @ B.double().abs().transpose(1, 2)
        mx = ((out - ref).abs() / sumabs).max().item()
        cub = ((A.cuda().float() @ B.cuda().float().transpose(1, 2)).cpu().double() - ref).norm() / ref.norm()
        print(f"| {K} | {rel_fro:.3g} | {rel_q:.3g} | {mx:.3g} | {cub.item():.3g} |")
        assert rel_q < bound


def test_tc_rejects_shapes_that_do_not_pair():
    m = _lib()
    A = _rand((1, 128, 128), 12)
    B = _rand((1, 256, 128), 13)
    with pytest.raises(m.MuonError):
        m.debug_gemm(A, B)
