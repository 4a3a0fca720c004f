"""GPU parity of convrot_linear_act_pack: the linear with an activation whose
epilogue also applies the next linear's rotation and row absmax, followed by a
light quantize launch ("Runtime activation quantization" of the page "INT8
Convrot Safetensors" applied to the hidden activations H of a DiT MLP).

The reference is the oracle's pack of H, where H comes from convrot_linear_act
on the same codes: the fused epilogue computes the same H bit for bit before
rotating it, so the codes and scales must agree with the oracle under the same
rules as the standalone pack (tests/parity.py)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from int8_hadamard_rotated_convrot_gb300 import convrot as cr  # noqa: E402
from int8_hadamard_rotated_convrot_gb300 import inputs  # noqa: E402

from . import parity  # noqa: E402


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


def codes_np(p):
    return p.codes_as_int8().cpu().numpy().astype(np.int32)


def check_against_oracle(H, p, G):
    Q, s, v = oracle.pack_rows(H, G)
    parity.check_scales(p.scale.cpu().numpy(), s)
    return parity.check_codes(codes_np(p), Q, v)


@pytest.mark.parametrize("out_codes", [cr.CODES_BF16, cr.CODES_I8], ids=["bf16-out", "i8-out"])
@pytest.mark.parametrize("m,k,n,G,act", [(300, 512, 768, 256, 1), (300, 512, 768, 64, 2), (129, 256, 512, 16, 0),
                                         (64, 256, 1024, 4, 1), (520, 1024, 2048, 256, 0), (300, 512, 1024, 1024, 1),
                                         (200, 256, 320, 64, 1)],
                         ids=["G256-erf", "G64-tanh", "G16-plain-m129", "G4-m64", "G256-plain", "G1024-fallback",
                              "n320-fallback"])
def test_linear_act_pack_matches_oracle_pack_of_h(m, k, n, G, act, out_codes):
    """Fused form (bf16 codes, n % 256 == 0, G <= 256) and the two-launch form for
    the other shapes, with canaries around the packed output."""
    rng = np.random.default_rng(m + k + n + G + act)
    X = rng.standard_normal((m, k)).astype(np.float32)
    X[:, rng.choice(k, 2, replace=False)] *= 50
    W = (0.05 * rng.standard_normal((n, k))).astype(np.float32)
    b = (0.1 * rng.standard_normal(n)).astype(np.float32)
    px = cr.convrot_pack_activations(to_dev(X), 64, cr.CODES_BF16)
    pw = cr.convrot_quantize_weights(to_dev(W), 64, cr.CODES_BF16)
    H = cr.convrot_linear_act(px, pw, to_dev(b), act)
    ldq = cr.convrot_ldq(n) + 64
    dtype = torch.int8 if out_codes == cr.CODES_I8 else torch.bfloat16
    fill = 90 if out_codes == cr.CODES_I8 else 3.0
    qbig = torch.full((m + 2, ldq), fill, dtype=dtype, device="cuda")
    sbig = torch.full((m + 1,), -7.0, dtype=torch.float32, device="cuda")
    out = cr.Packed(qbig[:m], sbig[:m], m, n, 0, out_codes)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cr.convrot_linear_act_pack(px, pw, to_dev(b), act, G, out_codes, out=out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == cr.OK
    assert (out.rows, out.k, out.group_size) == (m, n, G)
    kpad = cr.convrot_ldq(n)
    assert torch.all(qbig[:m, kpad:] == fill) and torch.all(qbig[m:] == fill) and float(sbig[m]) == -7.0
    assert torch.all(qbig[:m, n:kpad] == 0)
    check_against_oracle(H.cpu().numpy(), out, G)


def test_linear_act_pack_rejects_bad_requests():
    rng = np.random.default_rng(3)
    px = cr.convrot_pack_activations(to_dev(rng.standard_normal((8, 256)).astype(np.float32)), 64, cr.CODES_BF16)
    pw = cr.convrot_quantize_weights(to_dev(rng.standard_normal((512, 256)).astype(np.float32)), 64, cr.CODES_BF16)
    with pytest.raises(ValueError):  # too small a workspace
        cr.convrot_linear_act_pack(px, pw, None, 0, 256, work=torch.empty(16, dtype=torch.uint8, device="cuda"))
    with pytest.raises(cr.ConvrotError) as e:  # G does not divide n
        cr.convrot_linear_act_pack(px, pw, None, 0, 1024)
    assert e.value.status == cr.ERR_GROUP_SIZE


@pytest.mark.slow
def test_full_size_mlp_pair_fused_pack():
    """The DiT MLP pair with the down projection's pack fused into the up
    projection (M4096: K3072 -> N12288, GELU erf form, G256 -> N3072), as the bench
    runs it: the hidden activations' codes and scales on every row against the
    oracle's pack of H (H from the unfused linear, bit for bit the same), then the
    down projection from those codes on 520 sampled rows."""
    wl = inputs.WORKLOADS["mlp_pair"]
    G, bf16 = wl.G, cr.CODES_BF16
    X = inputs.activations(wl)
    (Wu,), bu = inputs.stage_weights(wl, 0)
    (Wd,), bd = inputs.stage_weights(wl, 1)
    px = cr.convrot_pack_activations(to_dev(X), G, bf16)
    pu = cr.convrot_quantize_weights(to_dev(Wu), G, bf16)
    pdn = cr.convrot_quantize_weights(to_dev(Wd), G, bf16)
    ph = cr.empty_packed(wl.m, wl.n, bf16, "cuda")
    ph.scale.fill_(float("nan"))
    cr.convrot_linear_act_pack(px, pu, to_dev(bu), wl.act, G, bf16, out=ph)
    Y = cr.convrot_linear(ph, pdn, to_dev(bd), out=torch.full((wl.m, wl.down_n), float("nan"), device="cuda"))
    H = cr.convrot_linear_act(px, pu, to_dev(bu), wl.act)
    torch.cuda.synchronize()
    assert not torch.isnan(Y).any() and not torch.isnan(ph.scale).any()
    H_np = H.cpu().numpy()
    del H
    flips = 0
    s_all, q_all = ph.scale.cpu().numpy(), codes_np(ph)
    for r0 in range(0, wl.m, 1024):
        Qc, sc, vc = oracle.pack_rows(H_np[r0:r0 + 1024], G)
        parity.check_scales(s_all[r0:r0 + 1024], sc)
        flips += parity.check_codes(q_all[r0:r0 + 1024], Qc, vc)
    rows = np.unique(np.concatenate([np.random.default_rng(99).choice(wl.m - 8, 512, replace=False),
                                     np.arange(wl.m - 8, wl.m)]))
    Qd_ref, sd_ref, _ = oracle.pack_rows(Wd, G, want_pre_round=False)
    qd_gpu, sd_gpu = codes_np(pdn), pdn.scale.cpu().numpy()
    qh_rows, sh_rows = q_all[rows], s_all[rows]
    Y_rows = Y[torch.from_numpy(rows).cuda()].cpu().numpy()
    A2 = oracle.gemm_i32(qh_rows.astype(np.int8), qd_gpu.astype(np.int8), wl.n)
    _, Y64 = oracle.reconstruct(A2, sh_rows, sd_gpu, bd)
    parity.check_y_same_codes(Y_rows, Y64, A2, sh_rows, sd_gpu, bd)
    Qh_ref, sh_ref, _ = oracle.pack_rows(H_np[rows], G, want_pre_round=False)
    _, Y64_ref = oracle.reconstruct(oracle.gemm_i32(Qh_ref, Qd_ref, wl.n), sh_ref, sd_ref, bd)
    e3 = parity.check_y_end_to_end(Y_rows, Y64_ref, (qh_rows, Qh_ref), (qd_gpu, Qd_ref), sh_rows, sd_gpu)
    parity.record("mlp_pair, pack fused into the up projection (down, from the fused codes)", y_rows=int(rows.size),
                  qh_flips_all_rows=flips, **e3)
