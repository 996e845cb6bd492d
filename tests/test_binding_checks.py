"""The Python binding refuses operands whose shape or dtype the C side could
not check (it sees only pointers): each case raises MxsError before anything
reaches a device.  CPU tensors serve here; the checks come first."""
import pytest

torch = pytest.importorskip("torch")

import mxfp4_speculative_verification_gb300 as mxs  # noqa: E402


def _gemm_operands(M=5, N=64, K=128):
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    nib = torch.zeros((N, K // 2), dtype=torch.uint8)
    sc = torch.zeros((N, K // 32), dtype=torch.uint8)
    return x, nib, sc


@pytest.mark.parametrize("fn", [mxs.mxfp4_verify_gemm, mxs.mxfp4_verify_gemm_noalloc])
def test_gemm_wrappers_reject_wrong_weight_shapes(fn):
    x, nib, sc = _gemm_operands()
    with pytest.raises(mxs.MxsError):
        fn(x, nib, sc[:, :3])                      # scales [N, K/32 - 1]: would be read past its end
    with pytest.raises(mxs.MxsError):
        fn(x, nib[:, :10], sc)                     # nibbles too short
    with pytest.raises(mxs.MxsError):
        fn(x.float(), nib, sc)                     # x not bf16
    with pytest.raises(mxs.MxsError):
        fn(x, nib.to(torch.int16), sc)             # nibbles not uint8
    with pytest.raises(mxs.MxsError):
        fn(x[0], nib, sc)                          # x not 2-D


@pytest.mark.parametrize("fn", [mxs.mxfp4_verify_gemm, mxs.mxfp4_verify_gemm_noalloc])
def test_gemm_wrappers_reject_wrong_outputs(fn):
    x, nib, sc = _gemm_operands()
    with pytest.raises(mxs.MxsError):
        fn(x, nib, sc, out=torch.zeros((5, 63), dtype=torch.float32))   # would be written past its end
    with pytest.raises(mxs.MxsError):
        fn(x, nib, sc, out=torch.zeros((5, 64), dtype=torch.float16))   # wrong dtype
    with pytest.raises(mxs.MxsError):
        fn(x, nib, sc, dev_status=torch.zeros(1, dtype=torch.int64))


def test_spec_accept_rejects_wrong_outputs():
    B, K, V = 2, 3, 16
    p = torch.zeros((B, K + 1, V), dtype=torch.float32)
    q = torch.zeros((B, K, V), dtype=torch.float32)
    d = torch.zeros((B, K), dtype=torch.int32)
    u = torch.zeros((B, K + 1), dtype=torch.float32)
    with pytest.raises(mxs.MxsError):
        mxs.spec_accept(p, q, d, u, out_tokens=torch.zeros((B, K), dtype=torch.int32))
    with pytest.raises(mxs.MxsError):
        mxs.spec_accept(p, q, d, u, n_emitted=torch.zeros((B + 1,), dtype=torch.int32))
    with pytest.raises(mxs.MxsError):
        mxs.spec_accept(p, q, d, u, row_flags=torch.zeros((B,), dtype=torch.int64))
    with pytest.raises(mxs.MxsError):
        mxs.spec_accept(p, q, d[:, :2], u)


def test_pack_rejects_wrong_outputs():
    w = torch.zeros((4, 64), dtype=torch.float32)
    with pytest.raises(mxs.MxsError):
        mxs.mxfp4_pack(w, nibbles=torch.zeros((4, 31), dtype=torch.uint8))
    with pytest.raises(mxs.MxsError):
        mxs.mxfp4_pack(w, scales=torch.zeros((4, 2), dtype=torch.int8))
    with pytest.raises(mxs.MxsError):
        mxs.mxfp4_pack(torch.zeros((4, 48), dtype=torch.float32))


def test_grouped_plan_checks_its_problems_once_at_construction():
    x, nib, sc = _gemm_operands()
    y = torch.zeros((5, 64), dtype=torch.float32)
    with pytest.raises(mxs.MxsError):
        mxs.GroupedGemm([])
    with pytest.raises(mxs.MxsError):
        mxs.GroupedGemm([(x, nib, sc[:, :3], y)])                            # scales too short
    with pytest.raises(mxs.MxsError):
        mxs.GroupedGemm([(x, nib, sc, torch.zeros((5, 63), dtype=torch.float32))])  # y too small
    with pytest.raises(mxs.MxsError):
        mxs.GroupedGemm([(x, nib, sc, y)])                                   # CPU tensors: no device launch
