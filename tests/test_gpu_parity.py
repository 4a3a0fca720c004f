"""GPU parity: the CUDA path through the C ABI against the oracle.

Tolerances are those of tests/parity.py. Small cases compare every element;
the full DiT-shaped workloads compare sampled rows the oracle can compute
quickly, plus the ragged tail rows, in the launch configuration bench.py uses.
"""

import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from int8_hadamard_rotated_convrot_gb300 import convrot as cr  # noqa: E402
from int8_hadamard_rotated_convrot_gb300 import inputs  # noqa: E402

from . import parity  # noqa: E402

CODES = [cr.CODES_I8, cr.CODES_BF16]
CODE_IDS = ["i8", "bf16"]
GEMM_CODES = [cr.CODES_I8, cr.CODES_BF16]
GEMM_IDS = ["i8", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_hadamard_rotated_convrot_gb300 import build

    build.build()
    cr.load()
    yield
    torch.cuda.synchronize()


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def codes_np(p: cr.Packed) -> np.ndarray:
    return p.codes_as_int8().cpu().numpy().astype(np.int32)


def special_rows(rng, m, k):
    X = rng.standard_normal((m, k)).astype(np.float32)
    X[:, rng.choice(k, size=max(1, k // 1000), replace=False)] *= 50
    X[0] = 0.0                      # zero row -> scale 0, codes 0
    if m > 1:
        X[1] = 0.0
        X[1, k // 3] = 1e4          # one spike spread over its group
    if m > 2:
        X[2] = 0.75                 # constant row: rotation output is exact
    if m > 3:
        X[3] *= 1e20                # huge but finite
    if m > 4:
        X[4] *= 1e-20               # tiny
    return X


def gpu_pack(X_np, G, codes, ldx_extra=4, canary=True):
    m, k = X_np.shape
    ldx = k + ldx_extra
    Xbig = np.zeros((m, ldx), np.float32)
    Xbig[:, :k] = X_np
    Xd = to_dev(Xbig)[:, :k]
    ldq = cr.convrot_ldq(k) + (64 if canary else 0)
    dtype = torch.int8 if codes == cr.CODES_I8 else torch.bfloat16
    fill = 90 if codes == cr.CODES_I8 else 3.0
    qbig = torch.full((m + 2, ldq), fill, dtype=dtype, device="cuda")
    sbig = torch.full((m + 1,), -7.0, dtype=torch.float32, device="cuda")
    out = cr.Packed(qbig[:m], sbig[:m], m, k, 0, codes)
    cr.convrot_pack_activations(Xd, G, codes, out=out)
    torch.cuda.synchronize()
    kpad = cr.convrot_ldq(k)
    # nothing outside [m, kpad) and the m scales was written; the pad is zero
    assert torch.all(qbig[:m, kpad:] == fill)
    assert torch.all(qbig[m:] == fill)
    assert float(sbig[m]) == -7.0
    assert torch.all(qbig[:m, k:kpad] == 0)
    return out


@pytest.mark.parametrize("codes", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("G,k", [(4, 3072), (16, 3072), (64, 3072), (256, 3072), (1024, 3072),
                                 (4096, 8192), (16, 400), (64, 192), (4, 4), (256, 256)])
def test_pack_matches_oracle(G, k, codes):
    rng = np.random.default_rng(G * 7 + k)
    m = 37
    X = special_rows(rng, m, k)
    p = gpu_pack(X, G, codes)
    Q, s, v = oracle.pack_rows(X, G)
    parity.check_scales(p.scale.cpu().numpy(), s)
    parity.check_codes(codes_np(p), Q, v)
    assert float(p.scale[0]) == 0.0 and torch.all(p.q[0, :cr.convrot_ldq(k)] == 0)


@pytest.mark.parametrize("G,k,m", [(256, 768, 3000), (4, 768, 3000), (64, 16384, 700), (256, 28672, 40),
                                   (1024, 3072, 3000), (1024, 16384, 500), (1024, 28672, 40),
                                   (1024, 1024, 999), (1024, 2048, 777), (1024, 5120, 301)],
                         ids=["ring-wraps", "ring-wraps-G4", "ring-one-cta-per-sm", "direct",
                              "G1024-ring", "G1024-ring-one-cta", "G1024-direct",
                              "G1024-ring-4-row-stages", "G1024-ring-2-row-stages", "G1024-ring-k5120"])
@pytest.mark.parametrize("codes", CODES, ids=CODE_IDS)
def test_pack_launch_forms(G, k, m, codes):
    """Each launch form of the G <= 1024 pack: a shared-memory ring that wraps many
    times, a ring of one CTA per SM (long rows), and the direct form. G = 1024
    uses 16-lane tiles; in the ring it takes the two-phase rotation (64-element
    chunks written back in place, then the tile layout), here with 1-, 2- and
    4-row stages and 2 or 3 stages."""
    rng = np.random.default_rng(G + k + m)
    X = special_rows(rng, m, k)
    p = gpu_pack(X, G, codes)
    Q, s, v = oracle.pack_rows(X, G)
    parity.check_scales(p.scale.cpu().numpy(), s)
    parity.check_codes(codes_np(p), Q, v)


@pytest.mark.parametrize("k", [4, 64, 256, 768, 1024, 2048, 3072, 4096, 5120, 8192, 12288, 16384, 20480, 24576,
                               28672])
@pytest.mark.parametrize("G", [4, 16, 256])
def test_pack_ring_shapes(G, k):
    """Every ring shape the launch picks by row length (four-lane layout: five
    one-stage CTAs per SM, or two or one CTA with two or more stages; eight-lane
    layout for G <= 16: four, two or one CTA) and the direct form past the rings
    (k = 28672), on 301 rows."""
    if k % G:
        pytest.skip("G must divide k")
    rng = np.random.default_rng(G * 131 + k)
    X = special_rows(rng, 301, k)
    p = gpu_pack(X, G, cr.CODES_BF16)
    Q, s, v = oracle.pack_rows(X, G)
    parity.check_scales(p.scale.cpu().numpy(), s)
    parity.check_codes(codes_np(p), Q, v)


def test_pack_hand_worked_rows(golden_dir):
    cases = json.load(open(os.path.join(golden_dir, "hand_worked_rows.json")))["rows"]
    for c in cases:
        for codes in CODES:
            X = np.array([c["x"]], np.float32)
            p = gpu_pack(X, c["G"], codes)
            num, den = c["scale_over"]
            assert float(p.scale[0]) == float(np.float32(num / den)), c["why"]
            np.testing.assert_array_equal(codes_np(p)[0], np.array(c["Q"]), err_msg=c["why"])


@pytest.mark.parametrize("G,k", [(256, 65536), (1024, 133120), (4, 131072), (4096, 131072)])
def test_pack_long_rows_use_clusters(G, k):
    rng = np.random.default_rng(k + G)
    X = special_rows(rng, 3, k)
    p = gpu_pack(X, G, cr.CODES_I8)
    Q, s, v = oracle.pack_rows(X, G)
    parity.check_scales(p.scale.cpu().numpy(), s)
    parity.check_codes(codes_np(p), Q, v)


@pytest.mark.parametrize("codes", CODES, ids=CODE_IDS)
@pytest.mark.parametrize("G,k,m", [(16384, 16384, 37), (16384, 49152, 9), (16384, 131072, 5), (65536, 65536, 9),
                                   (65536, 131072, 5)])
def test_pack_large_groups(G, k, m, codes):
    """G = 16384 and 65536 (4^7, 4^8): one CTA of four 4096-element blocks per
    16384 elements, the digits above the block across warps and, for 65536,
    across four CTAs of the row's cluster."""
    rng = np.random.default_rng(G + k + m)
    X = special_rows(rng, m, k)
    p = gpu_pack(X, G, codes)
    Q, s, v = oracle.pack_rows(X, G)
    parity.check_scales(p.scale.cpu().numpy(), s)
    parity.check_codes(codes_np(p), Q, v)
    assert float(p.scale[0]) == 0.0


def test_linear_end_to_end_group_16384():
    """The linear on rows packed with G = 16384 against the oracle end to end."""
    rng = np.random.default_rng(16384)
    m, k, n, G = 200, 16384, 256, 16384
    X = special_rows(rng, m, k)
    W = (0.02 * rng.standard_normal((n, k))).astype(np.float32)
    b = (0.01 * rng.standard_normal(n)).astype(np.float32)
    px = cr.convrot_pack_activations(to_dev(X), G, cr.CODES_BF16)
    pw = cr.convrot_quantize_weights(to_dev(W), G, cr.CODES_BF16)
    Y = cr.convrot_linear(px, pw, to_dev(b))
    torch.cuda.synchronize()
    ref = oracle.linear(X, W, b, G)
    Qw_ref, _, vw = oracle.pack_rows(W, G)
    parity.check_codes(codes_np(pw), Qw_ref, vw)
    e2e = parity.check_y_end_to_end(Y.cpu().numpy(), ref["Y64"], (codes_np(px), ref["Qx"]), (codes_np(pw), Qw_ref),
                                    px.scale.cpu().numpy(), pw.scale.cpu().numpy())
    parity.record("G = 16384, 200x16384x256", y_rows=m, **e2e)


def test_quantize_weights_equals_pack():
    rng = np.random.default_rng(5)
    W = (0.02 * rng.standard_normal((300, 512))).astype(np.float32)
    Wd = to_dev(W)
    a = cr.convrot_quantize_weights(Wd, 256)
    b = cr.convrot_pack_activations(Wd, 256)
    torch.cuda.synchronize()
    assert torch.equal(a.q, b.q) and torch.equal(a.scale, b.scale)
    Q, s, v = oracle.pack_rows(W, 256)
    parity.check_scales(a.scale.cpu().numpy(), s)
    parity.check_codes(codes_np(a), Q, v)


def test_empty_pack_and_linear():
    X = torch.empty((0, 256), dtype=torch.float32, device="cuda")
    p = cr.convrot_pack_activations(X, 256)
    w = cr.convrot_quantize_weights(torch.randn(8, 256, device="cuda"), 256)
    Y = cr.convrot_linear(p, w)
    torch.cuda.synchronize()
    assert Y.shape == (0, 8)


def test_empty_lora_and_fused_pack():
    """m == 0 is a no-op for the LoRA calls and the fused linear + pack as well."""
    X = torch.empty((0, 256), dtype=torch.float32, device="cuda")
    p = cr.convrot_pack_activations(X, 256, cr.CODES_BF16)  # (the LoRA chunk runs with bf16 codes)
    w = cr.convrot_quantize_weights(torch.randn(256, 256, device="cuda"), 256, cr.CODES_BF16)
    A_ext = cr.convrot_lora_prepare_down(0.05 * torch.randn(16, 256, device="cuda"))
    T = cr.convrot_lora_down(X, A_ext)
    assert T.shape == (0, cr.lora_cols(16))
    B_ext = cr.convrot_lora_prepare(0.02 * torch.randn(256, 16, device="cuda"), 2.0)
    Y = cr.convrot_linear_lora(p, w, None, cr.ACT_NONE, T, B_ext, 16)
    assert Y.shape == (0, 256)
    Y2 = cr.convrot_linear_lora_noalloc(p, w, None, cr.ACT_NONE, X, A_ext, B_ext, 16)
    assert Y2.shape == (0, 256)
    h = cr.convrot_linear_act_pack(p, w, None, cr.ACT_GELU_ERF, 256)
    assert (h.rows, h.k) == (0, 256)
    torch.cuda.synchronize()


@pytest.mark.parametrize("act", [cr.ACT_GELU_ERF, cr.ACT_GELU_TANH], ids=["gelu_erf", "gelu_tanh"])
@pytest.mark.parametrize("codes", GEMM_CODES, ids=GEMM_IDS)
@pytest.mark.parametrize("m,n,k", [(200, 300, 640), (64, 1000, 256), (300, 512, 1024)])
def test_linear_act_identical_codes(m, n, k, codes, act):
    """GELU fused into the epilogue, on both GEMM kernels; N = 300 and 1000 end
    in a ragged 32-column box."""
    rng = np.random.default_rng(m + n + k + act)
    Qx, Qw = random_codes(rng, m, k), random_codes(rng, n, k)
    sx = rng.uniform(0.0001, 0.002, m).astype(np.float32)
    sw = rng.uniform(0.0001, 0.002, n).astype(np.float32)
    b = rng.standard_normal(n).astype(np.float32)
    px = cr.packed_from_codes(to_dev(Qx), to_dev(sx), 64, codes)
    pw = cr.packed_from_codes(to_dev(Qw), to_dev(sw), 64, codes)
    Ybig = torch.full((m + 1, (n + 7) // 4 * 4), -3.0, dtype=torch.float32, device="cuda")
    Y = cr.convrot_linear_act(px, pw, to_dev(b), act, out=Ybig[:m, :n])
    torch.cuda.synchronize()
    A_ref = oracle.gemm_i32(Qx, Qw, k)
    _, Y64 = oracle.reconstruct(A_ref, sx, sw, b, act)
    parity.check_y_act_same_codes(Y.cpu().numpy(), Y64, A_ref, sx, sw, b)
    assert torch.all(Ybig[m:] == -3.0) and torch.all(Ybig[:, n:] == -3.0)
    # the values span GELU's curved part, not only its linear tails
    pre = oracle.reconstruct(A_ref, sx, sw, b)[1]
    assert (np.abs(pre) < 2).mean() > 0.2


def test_mlp_pair_stage_by_stage():
    """A DiT MLP: pack X, up projection with GELU in the epilogue, pack its
    output, down projection. Each stage is checked against the oracle given the
    GPU's own input to that stage."""
    rng = np.random.default_rng(77)
    m, d, h, G = 300, 512, 2048, 256
    X = special_rows(rng, m, d)
    Wu = (0.05 * rng.standard_normal((h, d))).astype(np.float32)
    bu = (0.1 * rng.standard_normal(h)).astype(np.float32)
    Wd = (0.02 * rng.standard_normal((d, h))).astype(np.float32)
    bd = (0.1 * rng.standard_normal(d)).astype(np.float32)
    px = cr.convrot_pack_activations(to_dev(X), G, cr.CODES_BF16)
    pu = cr.convrot_quantize_weights(to_dev(Wu), G, cr.CODES_BF16)
    pdn = cr.convrot_quantize_weights(to_dev(Wd), G, cr.CODES_BF16)
    H = cr.convrot_linear_act(px, pu, to_dev(bu), cr.ACT_GELU_ERF)
    ph = cr.convrot_pack_activations(H, G, cr.CODES_BF16)
    Y = cr.convrot_linear(ph, pdn, to_dev(bd))
    torch.cuda.synchronize()
    H_np = H.cpu().numpy()
    # stage 1: up projection + GELU against the oracle end to end
    ref1 = oracle.linear(X, Wu, bu, G, act=1)
    Qu_ref, _, _ = oracle.pack_rows(Wu, G, want_pre_round=False)
    parity.check_y_end_to_end(H_np, ref1["Y64"], (codes_np(px), ref1["Qx"]), (codes_np(pu), Qu_ref),
                              px.scale.cpu().numpy(), pu.scale.cpu().numpy())
    # stage 2: the pack of the GPU's hidden activations
    Qh_ref, sh_ref, vh = oracle.pack_rows(H_np, G)
    parity.check_scales(ph.scale.cpu().numpy(), sh_ref)
    parity.check_codes(codes_np(ph), Qh_ref, vh)
    # stage 3: down projection against the oracle from the same hidden activations
    ref3 = oracle.linear(H_np, Wd, bd, G)
    Qd_ref, _, _ = oracle.pack_rows(Wd, G, want_pre_round=False)
    parity.check_y_end_to_end(Y.cpu().numpy(), ref3["Y64"], (codes_np(ph), ref3["Qx"]), (codes_np(pdn), Qd_ref),
                              ph.scale.cpu().numpy(), pdn.scale.cpu().numpy())


def random_codes(rng, rows, k, sat=False):
    if sat:
        return np.where(rng.random((rows, k)) < 0.5, -127, 127).astype(np.int8)
    return rng.integers(-127, 128, size=(rows, k), dtype=np.int8)


@pytest.mark.parametrize("codes", GEMM_CODES, ids=GEMM_IDS)
@pytest.mark.parametrize("m,n,k,G", [(200, 300, 640, 64), (1, 1, 4, 4), (129, 257, 192, 64),
                                     (256, 384, 3072, 256), (37, 1000, 1024, 1024)])
def test_gemm_identical_codes_bit_exact(m, n, k, G, codes):
    rng = np.random.default_rng(m * n + k)
    Qx, Qw = random_codes(rng, m, k), random_codes(rng, n, k)
    sx = rng.uniform(0.001, 1.0, m).astype(np.float32)
    sw = rng.uniform(0.0001, 0.01, n).astype(np.float32)
    sx[0] = 0.0
    b = rng.standard_normal(n).astype(np.float32)
    px = cr.packed_from_codes(to_dev(Qx), to_dev(sx), G, codes)
    pw = cr.packed_from_codes(to_dev(Qw), to_dev(sw), G, codes)
    A = cr.convrot_gemm_i32(px, pw)
    Ybig = torch.full((m + 1, (n + 7) // 4 * 4), -3.0, dtype=torch.float32, device="cuda")
    Y = cr.convrot_linear(px, pw, to_dev(b), out=Ybig[:m, :n])
    torch.cuda.synchronize()
    A_ref = oracle.gemm_i32(Qx, Qw, k)
    np.testing.assert_array_equal(A.cpu().numpy(), A_ref)
    _, Y64 = oracle.reconstruct(A_ref, sx, sw, b)
    parity.check_y_same_codes(Y.cpu().numpy(), Y64, A_ref, sx, sw, b)
    assert torch.all(Ybig[m:] == -3.0) and torch.all(Ybig[:, n:] == -3.0)
    # no bias
    Y0 = cr.convrot_linear(px, pw)
    torch.cuda.synchronize()
    _, Y64n = oracle.reconstruct(A_ref, sx, sw, None)
    parity.check_y_same_codes(Y0.cpu().numpy(), Y64n, A_ref, sx, sw, None)


@pytest.mark.parametrize("codes", GEMM_CODES, ids=GEMM_IDS)
@pytest.mark.parametrize("m,n,act", [(512, 10240, 0), (512, 13468, 2), (300, 10112, 1), (512, 9984, 0),
                                     (768, 9984, 0)])
def test_gemm_split_last_wave_bit_exact(m, n, act, codes):
    """Shapes whose last, partial wave of 256 x 256 tiles is split along N
    into items, on a 152-SM GB300: 80 tiles (4 past 76 pairs: 32-wide items),
    106 tiles (30 past: 128-wide items, the ragged last column of tiles among
    them), 80 tiles with ragged M, 78 tiles (2 past: 32-wide items), and 117
    tiles (41 past: too many to split, so whole tiles through the same last-
    wave loop). A is bit-exact and Y (with and without GELU) matches the
    oracle, canaries intact."""
    k = 320
    rng = np.random.default_rng(m + n + act)
    Qx, Qw = random_codes(rng, m, k), random_codes(rng, n, k)
    sx = rng.uniform(0.001, 1.0, m).astype(np.float32)
    sw = rng.uniform(0.0001, 0.01, n).astype(np.float32)
    b = rng.standard_normal(n).astype(np.float32)
    px = cr.packed_from_codes(to_dev(Qx), to_dev(sx), 64, codes)
    pw = cr.packed_from_codes(to_dev(Qw), to_dev(sw), 64, codes)
    Abig = torch.full((m + 1, (n + 7) // 4 * 4), -5, dtype=torch.int32, device="cuda")
    A = cr.convrot_gemm_i32(px, pw, out=Abig[:m, :n])
    Ybig = torch.full((m + 1, (n + 7) // 4 * 4), -3.0, dtype=torch.float32, device="cuda")
    Y = cr.convrot_linear_act(px, pw, to_dev(b), act, out=Ybig[:m, :n])
    torch.cuda.synchronize()
    A_ref = oracle.gemm_i32(Qx, Qw, k)
    np.testing.assert_array_equal(A.cpu().numpy(), A_ref)
    assert torch.all(Abig[m:] == -5) and torch.all(Abig[:, n:] == -5)
    assert torch.all(Ybig[m:] == -3.0) and torch.all(Ybig[:, n:] == -3.0)
    _, Y64 = oracle.reconstruct(A_ref, sx, sw, b, act)
    check = parity.check_y_act_same_codes if act else parity.check_y_same_codes
    check(Y.cpu().numpy(), Y64, A_ref, sx, sw, b)


@pytest.mark.parametrize("codes", GEMM_CODES, ids=GEMM_IDS)
@pytest.mark.parametrize("k,G", [(12288, 256), (133144, 4)])
def test_gemm_saturated_int32_headroom(codes, k, G):
    """All-+-127 codes: |A| reaches 16129 * k, 198,193,152 at k = 12288 and, at the
    largest k the ABI accepts (133144, 131 exact fp32 chunks on the tensor-core
    path), 2,147,479,576: 4,071 below the int32 limit."""
    rng = np.random.default_rng(1)
    m, n = 130, 136
    Qx = random_codes(rng, m, k, sat=True)
    Qw = random_codes(rng, n, k, sat=True)
    Qx[0] = 127
    Qw[0] = 127
    Qw[1] = -127
    px = cr.packed_from_codes(to_dev(Qx), torch.ones(m, device="cuda"), G, codes)
    pw = cr.packed_from_codes(to_dev(Qw), torch.ones(n, device="cuda"), G, codes)
    A = cr.convrot_gemm_i32(px, pw).cpu().numpy()
    A_ref = oracle.gemm_i32(Qx, Qw, k)
    assert A_ref[0, 0] == 16129 * k and A_ref[0, 1] == -16129 * k
    np.testing.assert_array_equal(A, A_ref)


@pytest.mark.parametrize("codes", GEMM_CODES, ids=GEMM_IDS)
def test_linear_end_to_end_tiny(codes):
    wl = inputs.WORKLOADS["tiny"]
    X, W, b = inputs.activations(wl), inputs.weights(wl), inputs.bias(wl)
    px = cr.convrot_pack_activations(to_dev(X), wl.G, codes)
    pw = cr.convrot_quantize_weights(to_dev(W), wl.G, codes)
    Y = cr.convrot_linear(px, pw, to_dev(b))
    A = cr.convrot_gemm_i32(px, pw)
    torch.cuda.synchronize()
    ref = oracle.linear(X, W, b, wl.G)
    parity.check_scales(px.scale.cpu().numpy(), ref["sx"])
    parity.check_scales(pw.scale.cpu().numpy(), ref["sw"])
    parity.check_codes(codes_np(px), ref["Qx"], ref["vx"])
    Qw_ref, _, vw = oracle.pack_rows(W, wl.G)
    parity.check_codes(codes_np(pw), Qw_ref, vw)
    e2e = parity.check_y_end_to_end(Y.cpu().numpy(), ref["Y64"], (codes_np(px), ref["Qx"]),
                                    (codes_np(pw), Qw_ref), px.scale.cpu().numpy(), pw.scale.cpu().numpy())
    parity.record(f"tiny ({'i8' if codes == cr.CODES_I8 else 'bf16'} codes)", y_rows=wl.m, **e2e)
    # with the GPU's own codes the integer product and the epilogue are exact
    qx, qw = codes_np(px).astype(np.int8), codes_np(pw).astype(np.int8)
    A_ref = oracle.gemm_i32(qx, qw, wl.k)
    np.testing.assert_array_equal(A.cpu().numpy(), A_ref)
    sx, sw = px.scale.cpu().numpy(), pw.scale.cpu().numpy()
    _, Y64 = oracle.reconstruct(A_ref, sx, sw, b)
    parity.check_y_same_codes(Y.cpu().numpy(), Y64, A_ref, sx, sw, b)


FULL = ["attn_qkv", "mlp_up", "mlp_down", "sweep_G4", "sweep_G16", "sweep_G64", "sweep_G256", "sweep_G1024",
        "video_n5120", "video_n13824"]


def check_pack_all_rows(X, p: cr.Packed, G: int, chunk: int = 4096) -> int:
    """The pack against the oracle on every row, in chunks of rows: scales and codes.
    Returns how many codes differ (each one a tie the code rule allows)."""
    s_all, q_all = p.scale.cpu().numpy(), codes_np(p)
    flips = 0
    for r0 in range(0, X.shape[0], chunk):
        r1 = min(X.shape[0], r0 + chunk)
        Qc, sc, vc = oracle.pack_rows(X[r0:r1], G)
        parity.check_scales(s_all[r0:r1], sc)
        flips += parity.check_codes(q_all[r0:r1], Qc, vc)
    return flips


def sample_rows(m: int, n_rows: int, seed: int = 123) -> np.ndarray:
    """n_rows seeded random rows plus the last 8 (the ragged tail of the last tile)."""
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(m - 8, n_rows, replace=False), np.arange(m - 8, m)]))


@pytest.mark.slow
@pytest.mark.parametrize("name,codes", [(n, cr.CODES_BF16) for n in FULL] + [("mlp_up", cr.CODES_I8),
                                                                         ("mlp_down", cr.CODES_I8)],
                         ids=FULL + ["mlp_up-i8", "mlp_down-i8"])
def test_full_size_sampled(name, codes):
    """Full workload on the GPU in the bench's configuration: the pack against the
    oracle on every row, Y on sampled rows plus the tail. The I8 cases store the
    page's int8 codes and run the tensor-core kernel that widens them on chip."""
    wl = inputs.WORKLOADS[name]
    X, W, b = inputs.activations(wl), inputs.weights(wl), inputs.bias(wl)
    px = cr.convrot_pack_activations(to_dev(X), wl.G, codes)
    pw = cr.convrot_quantize_weights(to_dev(W), wl.G, codes)
    # NaN-filled output: a tile the GEMM skipped cannot pass for a stale correct one
    Y = cr.convrot_linear(px, pw, to_dev(b), out=torch.full((wl.m, wl.n), float("nan"), device="cuda"))
    torch.cuda.synchronize()
    assert not torch.isnan(Y).any()
    # the pack on every row, in chunks of rows: scales and codes against the oracle
    pack_flips = check_pack_all_rows(X, px, wl.G)
    # Y on 512 seeded random rows (256 on the largest shape) plus the tail rows
    rows = sample_rows(wl.m, 256 if wl.m * wl.n * wl.k > 2e12 else 512)
    Xs = X[rows]
    Qx_ref, sx_ref, vx = oracle.pack_rows(Xs, wl.G)
    Qw_ref, sw_ref, vw = oracle.pack_rows(W, wl.G)
    sx_gpu = px.scale.cpu().numpy()[rows]
    qx_gpu = codes_np(px)[rows]
    parity.check_scales(sx_gpu, sx_ref)
    parity.check_codes(qx_gpu, Qx_ref, vx)
    sw_gpu = pw.scale.cpu().numpy()
    qw_gpu = codes_np(pw)
    parity.check_scales(sw_gpu, sw_ref)
    w_flips = parity.check_codes(qw_gpu, Qw_ref, vw)
    del vw
    Y_rows = Y[torch.from_numpy(rows).cuda()].cpu().numpy()
    # same codes: exact integer product, epilogue within 1e-6
    A_gpu_codes = oracle.gemm_i32(qx_gpu.astype(np.int8), qw_gpu.astype(np.int8), wl.k)
    _, Y64 = oracle.reconstruct(A_gpu_codes, sx_gpu, sw_gpu, b)
    parity.check_y_same_codes(Y_rows, Y64, A_gpu_codes, sx_gpu, sw_gpu, b)
    # end to end against the oracle's own codes
    A_ref = oracle.gemm_i32(Qx_ref, Qw_ref, wl.k)
    _, Y64_ref = oracle.reconstruct(A_ref, sx_ref, sw_ref, b)
    e2e = parity.check_y_end_to_end(Y_rows, Y64_ref, (qx_gpu, Qx_ref), (qw_gpu, Qw_ref), sx_gpu, sw_gpu)
    parity.record(name + ("" if codes == cr.CODES_BF16 else " (I8 codes)"), qx_codes=int(wl.m * wl.k),
                  qx_flips_all_rows=pack_flips, qw_codes=int(wl.n * wl.k),
                  qw_flips=w_flips, y_rows=int(rows.size), **e2e)


def test_grouped_linears_share_one_pack():
    """q, k, v against one packed input in one GEMM equal three separate linears bit for bit."""
    rng = np.random.default_rng(31)
    m, k, sizes = 300, 512, (256, 384, 200)
    X = rng.standard_normal((m, k)).astype(np.float32)
    Ws = [(0.02 * rng.standard_normal((n, k))).astype(np.float32) for n in sizes]
    bs = [rng.standard_normal(n).astype(np.float32) for n in sizes]
    px = cr.convrot_pack_activations(to_dev(X), 64, cr.CODES_BF16)
    pw = cr.quantize_weights_grouped([to_dev(W) for W in Ws], 64, cr.CODES_BF16)
    Y = cr.convrot_linear(px, pw, to_dev(np.concatenate(bs)))
    singles = []
    for W, b in zip(Ws, bs):
        p1 = cr.convrot_quantize_weights(to_dev(W), 64, cr.CODES_BF16)
        singles.append(cr.convrot_linear(px, p1, to_dev(b)))
    torch.cuda.synchronize()
    for view, single in zip(cr.split_columns(Y, sizes), singles):
        assert torch.equal(view, single)
    # and against the oracle, end to end
    ref = oracle.linear(X, np.concatenate(Ws), np.concatenate(bs), 64)
    Qw_ref, _, _ = oracle.pack_rows(np.concatenate(Ws), 64, want_pre_round=False)
    parity.check_y_end_to_end(Y.cpu().numpy(), ref["Y64"], (codes_np(px), ref["Qx"]), (codes_np(pw), Qw_ref),
                              px.scale.cpu().numpy(), pw.scale.cpu().numpy())


@pytest.mark.slow
def test_full_size_attention_grouped_qkv():
    """The attention workload as the bench runs it: one pack, q/k/v in one grouped GEMM."""
    wl = inputs.WORKLOADS["attn_qkv"]
    X = inputs.activations(wl)
    Ws = [inputs.weights(wl, i) for i in range(3)]
    bs = [inputs.bias(wl, i) for i in range(3)]
    px = cr.convrot_pack_activations(to_dev(X), wl.G, cr.CODES_BF16)
    pw = cr.quantize_weights_grouped([to_dev(W) for W in Ws], wl.G, cr.CODES_BF16)
    Y = cr.convrot_linear(px, pw, to_dev(np.concatenate(bs)),
                          out=torch.full((wl.m, 3 * wl.n), float("nan"), device="cuda"))
    torch.cuda.synchronize()
    assert not torch.isnan(Y).any()
    rows = np.concatenate([np.random.default_rng(5).choice(wl.m - 8, 48, replace=False), np.arange(wl.m - 8, wl.m)])
    Qx_ref, sx_ref, vx = oracle.pack_rows(X[rows], wl.G)
    Qw_ref, sw_ref, _ = oracle.pack_rows(np.concatenate(Ws), wl.G, want_pre_round=False)
    A_ref = oracle.gemm_i32(Qx_ref, Qw_ref, wl.k)
    _, Y64 = oracle.reconstruct(A_ref, sx_ref, sw_ref, np.concatenate(bs))
    e2e = parity.check_y_end_to_end(Y[torch.from_numpy(rows).cuda()].cpu().numpy(), Y64,
                                    (codes_np(px)[rows], Qx_ref), (codes_np(pw), Qw_ref),
                                    px.scale.cpu().numpy()[rows], pw.scale.cpu().numpy())
    parity.record("attn_qkv grouped (N = 3 x 3072)", y_rows=int(rows.size), **e2e)


@pytest.mark.slow
def test_full_size_mlp_pair():
    """The DiT MLP pair as the bench runs it (M4096: K3072 -> N12288 with GELU (erf
    form) in the up projection's epilogue, pack of that output, -> N3072), into
    NaN-filled outputs. Stage by stage, each against the oracle given the GPU's own
    input to that stage: both packs on every row; the hidden activations and the
    output on 512 seeded rows plus the tail, with the GPU's codes (exact integer
    product, epilogue within its bound) and end to end from the oracle's codes."""
    wl = inputs.WORKLOADS["mlp_pair"]
    G, bf16 = wl.G, cr.CODES_BF16
    X = inputs.activations(wl)
    (Wu,), bu = inputs.stage_weights(wl, 0)
    (Wd,), bd = inputs.stage_weights(wl, 1)
    px = cr.convrot_pack_activations(to_dev(X), G, bf16)
    pu = cr.convrot_quantize_weights(to_dev(Wu), G, bf16)
    pdn = cr.convrot_quantize_weights(to_dev(Wd), G, bf16)
    H = cr.convrot_linear_act(px, pu, to_dev(bu), wl.act,
                              out=torch.full((wl.m, wl.n), float("nan"), device="cuda"))
    ph = cr.convrot_pack_activations(H, G, bf16)
    Y = cr.convrot_linear(ph, pdn, to_dev(bd), out=torch.full((wl.m, wl.down_n), float("nan"), device="cuda"))
    torch.cuda.synchronize()
    assert not torch.isnan(H).any() and not torch.isnan(Y).any()
    rows = sample_rows(wl.m, 512, seed=321)
    rows_d = torch.from_numpy(rows).cuda()
    stats = {"y_rows": int(rows.size)}
    # stage 1: pack X (every row), up projection + GELU (sampled rows)
    stats["qx_flips_all_rows"] = check_pack_all_rows(X, px, G)
    Qu_ref, su_ref, vu = oracle.pack_rows(Wu, G)
    qu_gpu, su_gpu = codes_np(pu), pu.scale.cpu().numpy()
    parity.check_scales(su_gpu, su_ref)
    stats["qw_up_flips"] = parity.check_codes(qu_gpu, Qu_ref, vu)
    del vu
    qx_rows, sx_rows = codes_np(px)[rows], px.scale.cpu().numpy()[rows]
    H_rows = H[rows_d].cpu().numpy()
    A1 = oracle.gemm_i32(qx_rows.astype(np.int8), qu_gpu.astype(np.int8), wl.k)
    _, H64 = oracle.reconstruct(A1, sx_rows, su_gpu, bu, wl.act)
    parity.check_y_act_same_codes(H_rows, H64, A1, sx_rows, su_gpu, bu)
    Qx_ref, sx_ref, _ = oracle.pack_rows(X[rows], G, want_pre_round=False)
    A1_ref = oracle.gemm_i32(Qx_ref, Qu_ref, wl.k)
    H_chain, H64_ref = oracle.reconstruct(A1_ref, sx_ref, su_ref, bu, wl.act)  # H_chain: fp32, as stored
    e1 = parity.check_y_end_to_end(H_rows, H64_ref, (qx_rows, Qx_ref), (qu_gpu, Qu_ref), sx_rows, su_gpu)
    parity.record("mlp_pair up + GELU (stage 1)", **stats, **e1)
    del A1, H64, A1_ref, H64_ref
    # stage 2: the pack of the GPU's hidden activations, every row
    H_np = H.cpu().numpy()
    ph_flips = check_pack_all_rows(H_np, ph, G, chunk=1024)
    # stage 3: down projection from the GPU's hidden activations (sampled rows)
    Qd_ref, sd_ref, vd = oracle.pack_rows(Wd, G)
    qd_gpu, sd_gpu = codes_np(pdn), pdn.scale.cpu().numpy()
    parity.check_scales(sd_gpu, sd_ref)
    qd_flips = parity.check_codes(qd_gpu, Qd_ref, vd)
    del vd
    qh_rows, sh_rows = codes_np(ph)[rows], ph.scale.cpu().numpy()[rows]
    Y_rows = Y[rows_d].cpu().numpy()
    A2 = oracle.gemm_i32(qh_rows.astype(np.int8), qd_gpu.astype(np.int8), wl.n)
    _, Y64 = oracle.reconstruct(A2, sh_rows, sd_gpu, bd)
    parity.check_y_same_codes(Y_rows, Y64, A2, sh_rows, sd_gpu, bd)
    Qh_ref, sh_ref, _ = oracle.pack_rows(H_np[rows], G, want_pre_round=False)
    A2_ref = oracle.gemm_i32(Qh_ref, Qd_ref, wl.n)
    _, Y64_ref = oracle.reconstruct(A2_ref, sh_ref, sd_ref, bd)
    e3 = parity.check_y_end_to_end(Y_rows, Y64_ref, (qh_rows, Qh_ref), (qd_gpu, Qd_ref), sh_rows, sd_gpu)
    # the whole chain in the oracle alone (its own hidden activations, rounded to fp32
    # as they are stored), against the GPU's output: recorded, not a tolerance rule
    Qc, sc, _ = oracle.pack_rows(H_chain, G, want_pre_round=False)
    _, Y64_chain = oracle.reconstruct(oracle.gemm_i32(Qc, Qd_ref, wl.n), sc, sd_ref, bd)
    chain = float(np.max(np.abs(Y_rows - Y64_chain)) / (1e-3 * np.max(np.abs(Y64_chain))))
    parity.record("mlp_pair down (stage 3, from the GPU's hidden activations)", y_rows=int(rows.size),
                  qh_flips_all_rows=ph_flips, qw_down_flips=qd_flips,
                  chain_max_err_over_plain=chain, **e3)


@pytest.mark.slow
def test_full_size_mlp_up_lora():
    """MLP up with the rank-64 runtime LoRA (scale 2) as the bench runs it: LoRA down
    from the unrotated X, pack, and the linear with the correction chunk, into
    NaN-filled outputs. The pack on every row; T and Y on 512 seeded rows plus the
    tail: T against the fp64 oracle within its split-TF32 bound, Y with the GPU's
    codes within the base-plus-correction bound, and end to end from the oracle's
    codes and correction."""
    wl = inputs.WORKLOADS["mlp_up_lora"]
    G, r, bf16 = wl.G, wl.lora_r, cr.CODES_BF16
    X = inputs.activations(wl)
    (W,), b = inputs.stage_weights(wl, 0)
    Al, Bl = inputs.lora_weights(wl)
    Xd = to_dev(X)
    A_ext = cr.convrot_lora_prepare_down(to_dev(Al))
    B_ext = cr.convrot_lora_prepare(to_dev(Bl), wl.lora_scale)
    pw = cr.convrot_quantize_weights(to_dev(W), G, bf16)
    T_ext = cr.convrot_lora_down(Xd, A_ext)
    px = cr.convrot_pack_activations(Xd, G, bf16)
    Y = cr.convrot_linear_lora(px, pw, to_dev(b), wl.act, T_ext, B_ext, r,
                               out=torch.full((wl.m, wl.n), float("nan"), device="cuda"))
    torch.cuda.synchronize()
    assert not torch.isnan(Y).any()
    flips = check_pack_all_rows(X, px, G)
    rows = sample_rows(wl.m, 512, seed=654)
    rows_d = torch.from_numpy(rows).cuda()
    Xs = X[rows]
    # T on the sampled rows
    t = T_ext[rows_d].float().cpu().numpy()
    T_ref, D = oracle.lora_delta(Xs, Al, Bl, wl.lora_scale)
    l1_t = np.abs(Xs.astype(np.float64)) @ np.abs(Al.astype(np.float64)).T
    parity.check_lora_t(t[:, :r].astype(np.float64) + t[:, 2 * r:3 * r], T_ref, l1_t, wl.k)
    # Y with the GPU's codes: exact integer product, correction within its bound
    Qw_ref, sw_ref, vw = oracle.pack_rows(W, G)
    qw_gpu, sw_gpu = codes_np(pw), pw.scale.cpu().numpy()
    parity.check_scales(sw_gpu, sw_ref)
    w_flips = parity.check_codes(qw_gpu, Qw_ref, vw)
    del vw
    qx_rows, sx_rows = codes_np(px)[rows], px.scale.cpu().numpy()[rows]
    Y_rows = Y[rows_d].cpu().numpy()
    A = oracle.gemm_i32(qx_rows.astype(np.int8), qw_gpu.astype(np.int8), wl.k)
    _, Y64 = oracle.reconstruct(A, sx_rows, sw_gpu, b, wl.act, add=D)
    l1 = wl.lora_scale * l1_t @ np.abs(Bl.astype(np.float64)).T
    parity.check_y_lora_same_codes(Y_rows, Y64, A, sx_rows, sw_gpu, b, l1, wl.k, r, wl.act)
    assert np.abs(D).mean() > 0.05 * np.abs(Y64).mean()  # the correction is not negligible
    # end to end from the oracle's codes and correction
    Qx_ref, sx_ref, _ = oracle.pack_rows(Xs, G, want_pre_round=False)
    _, Y64_ref = oracle.reconstruct(oracle.gemm_i32(Qx_ref, Qw_ref, wl.k), sx_ref, sw_ref, b, wl.act, add=D)
    e2e = parity.check_y_end_to_end(Y_rows, Y64_ref, (qx_rows, Qx_ref), (qw_gpu, Qw_ref), sx_rows, sw_gpu)
    parity.record("mlp_up_lora (r 64, scale 2)", y_rows=int(rows.size), qx_flips_all_rows=flips, qw_flips=w_flips,
                  **e2e)


def test_graph_replay_equals_eager_steps():
    """bench.py times its steps as one captured CUDA graph of the same C-ABI
    launches. Replaying it (pack, LoRA down, the LoRA linear with GELU, then
    the down-projection's pack and linear, on two rotating buffer sets) gives
    bit for bit what the eager calls give, and the status word stays clear."""
    rng = np.random.default_rng(31)
    m, k, n, r = 300, 512, 768, 32
    Xs = [to_dev(special_rows(rng, m, k)) for _ in range(2)]
    W1 = to_dev((0.02 * rng.standard_normal((n, k))).astype(np.float32))
    W2 = to_dev((0.02 * rng.standard_normal((k, n))).astype(np.float32))
    b1, b2 = to_dev(rng.standard_normal(n).astype(np.float32)), to_dev(rng.standard_normal(k).astype(np.float32))
    pw1, pw2 = cr.convrot_quantize_weights(W1, 64, cr.CODES_BF16), cr.convrot_quantize_weights(W2, 256, cr.CODES_BF16)
    A_ext = cr.convrot_lora_prepare_down(to_dev((0.05 * rng.standard_normal((r, k))).astype(np.float32)))
    B_ext = cr.convrot_lora_prepare(to_dev((0.05 * rng.standard_normal((n, r))).astype(np.float32)), 2.0)
    px1 = [cr.empty_packed(m, k, cr.CODES_BF16, "cuda") for _ in range(2)]
    px2 = [cr.empty_packed(m, n, cr.CODES_BF16, "cuda") for _ in range(2)]
    T = [torch.empty((m, cr.lora_cols(r)), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    H = [torch.empty((m, n), device="cuda") for _ in range(2)]
    Y = [torch.empty((m, k), device="cuda") for _ in range(2)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()

    def step(j):
        cr.convrot_lora_down(Xs[j], A_ext, out=T[j], dev_status=st, stream=s)
        cr.convrot_pack_activations(Xs[j], 64, cr.CODES_BF16, out=px1[j], dev_status=st, stream=s)
        cr.convrot_linear_lora(px1[j], pw1, b1, cr.ACT_GELU_TANH, T[j], B_ext, r, out=H[j], dev_status=st, stream=s)
        cr.convrot_pack_activations(H[j], 256, cr.CODES_BF16, out=px2[j], dev_status=st, stream=s)
        cr.convrot_linear_act(px2[j], pw2, b2, cr.ACT_NONE, out=Y[j], dev_status=st, stream=s)

    with torch.cuda.stream(s):
        for j in range(2):
            step(j)
    torch.cuda.synchronize()
    eager = [y.clone() for y in Y] + [h.clone() for h in H]
    for t in Y + H:
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for j in range(2):
            step(j)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, Y + H):
        assert torch.equal(a, b)
    assert int(st.item()) == cr.OK


# ---- runtime LoRA side branch

@pytest.mark.parametrize("m,k,r", [(300, 512, 16), (129, 3072, 64), (64, 200, 48), (1000, 1024, 256),
                                   (200, 1000, 96), (384, 2048, 176)])
def test_lora_down_against_oracle(m, k, r):
    """T = X A^T (three-term TF32 on tcgen05), stored as [hi | hi | lo | 0]."""
    rng = np.random.default_rng(m + k + r)
    X = special_rows(rng, m, k)
    A = (0.05 * rng.standard_normal((r, k))).astype(np.float32)
    cols = cr.lora_cols(r)
    Tbig = torch.full((m + 1, cols + 8), 7.0, dtype=torch.bfloat16, device="cuda")  # canaries
    A_ext = cr.convrot_lora_prepare_down(to_dev(A))
    ah, al = A_ext[:r, :k].cpu().numpy(), A_ext[r:, :k].cpu().numpy()
    np.testing.assert_array_equal(ah.astype(np.float64) + al, A.astype(np.float64))  # the split is exact
    assert np.all((ah.view(np.uint32) & 0x1fff) == 0)
    T_ext = cr.convrot_lora_down(to_dev(X), A_ext, out=Tbig[:m, :cols])
    torch.cuda.synchronize()
    t = T_ext.float().cpu().numpy()
    assert torch.all(Tbig[m:] == 7.0) and torch.all(Tbig[:, cols:] == 7.0)
    np.testing.assert_array_equal(t[:, :r], t[:, r:2 * r])
    assert np.all(t[:, 3 * r:] == 0.0)
    T_ref, _ = oracle.lora_delta(X, A, np.zeros((1, r), np.float32), 1.0)
    l1 = np.abs(X.astype(np.float64)) @ np.abs(A.astype(np.float64)).T
    parity.check_lora_t(t[:, :r].astype(np.float64) + t[:, 2 * r:3 * r], T_ref, l1, k)


@pytest.mark.parametrize("m,n,k,r,act", [(300, 300, 512, 32, 0), (300, 512, 1024, 64, 1), (64, 1000, 256, 16, 2),
                                         (513, 256, 3072, 128, 0), (512, 10240, 320, 64, 0),
                                         (512, 13468, 320, 32, 2)])
def test_linear_lora_identical_codes(m, n, k, r, act):
    """Y = act(A s_x s_w + b + scale (X A_l^T) B_l^T) with the LoRA term as an extra
    fp32 chunk of the pair GEMM (also for m <= 128, and for shapes whose last,
    partial wave is split along N into 32- and 128-wide items on a 152-SM GB300)."""
    rng = np.random.default_rng(m * 3 + n + k + r)
    X = special_rows(rng, m, k)
    Qx, Qw = random_codes(rng, m, k), random_codes(rng, n, k)
    sx = rng.uniform(0.0001, 0.002, m).astype(np.float32)
    sw = rng.uniform(0.0001, 0.002, n).astype(np.float32)
    b = rng.standard_normal(n).astype(np.float32)
    Al = (0.05 * rng.standard_normal((r, k))).astype(np.float32)
    Bl = (0.05 * rng.standard_normal((n, r))).astype(np.float32)
    scale = 2.0
    px = cr.packed_from_codes(to_dev(Qx), to_dev(sx), 64, cr.CODES_BF16)
    pw = cr.packed_from_codes(to_dev(Qw), to_dev(sw), 64, cr.CODES_BF16)
    T_ext = cr.convrot_lora_down(to_dev(X), cr.convrot_lora_prepare_down(to_dev(Al)))
    B_ext = cr.convrot_lora_prepare(to_dev(Bl), scale)
    Ybig = torch.full((m + 1, (n + 7) // 4 * 4), -3.0, dtype=torch.float32, device="cuda")
    Y = cr.convrot_linear_lora(px, pw, to_dev(b), act, T_ext, B_ext, r, out=Ybig[:m, :n])
    torch.cuda.synchronize()
    assert torch.all(Ybig[m:] == -3.0) and torch.all(Ybig[:, n:] == -3.0)
    A_ref = oracle.gemm_i32(Qx, Qw, k)
    _, D = oracle.lora_delta(X, Al, Bl, scale)
    _, Y64 = oracle.reconstruct(A_ref, sx, sw, b, act, add=D)
    l1 = scale * (np.abs(X.astype(np.float64)) @ np.abs(Al.astype(np.float64)).T) @ np.abs(Bl.astype(np.float64)).T
    parity.check_y_lora_same_codes(Y.cpu().numpy(), Y64, A_ref, sx, sw, b, l1, k, r, act)
    # the correction is not negligible next to the base output
    assert np.abs(D).mean() > 0.05 * np.abs(Y64).mean()


def test_lora_prepare_layout():
    rng = np.random.default_rng(9)
    n, r = 70, 48
    Bl = rng.standard_normal((n, r)).astype(np.float32)
    ext = cr.convrot_lora_prepare(to_dev(Bl), 1.5).float().cpu().numpy()
    v = 1.5 * Bl.astype(np.float64)
    hi, lo = ext[:, :r], ext[:, r:2 * r]
    np.testing.assert_array_equal(ext[:, 2 * r:3 * r], hi)
    assert np.all(ext[:, 3 * r:] == 0.0)
    assert np.all(np.abs(hi - v) <= 2.0 ** -8 * np.abs(v))          # hi is v rounded to bf16
    assert np.all(np.abs(hi + lo - v) <= 2.0 ** -16 * np.abs(v))    # hi + lo carries ~16 bits
