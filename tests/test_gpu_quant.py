"""GPU parity of tfd_quant_fp8 against the oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

from helpers import need_gpu
from oracle.quant import quant_fp8_block32, quant_fp8_row
from speculative_decoding_draft_row_gb300 import tfd
from synth import inputs

pytestmark = pytest.mark.gpu


def all_bf16_matrix(cols=4096):
    """Every finite bf16 bit pattern, 16 rows x 4096, with rows of very different amax."""
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32).copy()
    v[~np.isfinite(v)] = 0.0
    return v.reshape(-1, cols)


def gpu_quant(w_np, mode):
    w = torch.from_numpy(np.ascontiguousarray(w_np, dtype=np.float32)).to(torch.bfloat16).cuda()
    codes, scales = tfd.tfd_quant_fp8(w, mode)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("mode", [tfd.W_FP8_ROW, tfd.W_FP8_BLOCK32])
def test_every_bf16_value(mode):
    need_gpu()
    base = all_bf16_matrix()
    # tile with scaled copies so that every value meets many different scales
    with np.errstate(over="ignore"):
        w = np.concatenate([base, base * np.float32(2.0 ** -60), base[::-1] * np.float32(1.5),
                            base[:, ::-1] * np.float32(0.75)], axis=0)          # 64 rows
    w[~np.isfinite(w)] = 0.0
    w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()      # bf16-representable
    w[~np.isfinite(w)] = 0.0
    codes, scales = gpu_quant(w, mode)
    if mode == tfd.W_FP8_ROW:
        oc, os_ = quant_fp8_row(w)
        assert np.array_equal(scales.view(np.uint32), os_.view(np.uint32))
    else:
        oc, os_ = quant_fp8_block32(w)
        assert np.array_equal(scales, os_)
    assert np.array_equal(codes, oc)


@pytest.mark.parametrize("mode", [tfd.W_FP8_ROW, tfd.W_FP8_BLOCK32])
@pytest.mark.parametrize("shape", [(32, 16 * 3), (96, 4096), (4096, 4096 + 256 + 32), (64, 11008)])
def test_shapes_and_edges(mode, shape):
    need_gpu()
    n, k = shape
    if mode == tfd.W_FP8_BLOCK32 and (n % 32 or k % 32):
        pytest.skip("block form needs multiples of 32")
    w = inputs.normal_bf16((n, k), 0.02, 200).float().numpy()
    w[0] = 0.0                       # zero row / zero blocks
    w[1, ::3] = -0.0
    w[2] *= 1e4                      # large row
    w[3] *= 1e-30                    # tiny row
    w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()   # back onto bf16 values
    codes, scales = gpu_quant(w, mode)
    if mode == tfd.W_FP8_ROW:
        oc, os_ = quant_fp8_row(w)
        assert np.array_equal(scales.view(np.uint32), os_.view(np.uint32))
    else:
        oc, os_ = quant_fp8_block32(w)
        assert np.array_equal(scales, os_)
    assert np.array_equal(codes, oc)


@pytest.mark.parametrize("mode", [tfd.W_FP8_ROW, tfd.W_FP8_BLOCK32])
def test_full_head_sampled_rows(mode):
    """The full 163840 x 4096 head: bit-exact on 64 sampled 32-row blocks (2048 rows)."""
    need_gpu()
    w, _ = inputs.head(tie_frac=0.01)
    wd = w.cuda()
    codes, scales = tfd.tfd_quant_fp8(wd, mode)
    torch.cuda.synchronize()
    rng = np.random.default_rng([0, 201, 0])
    blocks = np.sort(rng.choice(163840 // 32, 64, replace=False))
    blocks[0], blocks[-1] = 0, 163840 // 32 - 1
    rows = (blocks[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    wr = w[torch.from_numpy(rows)].float().numpy()
    c_gpu = codes[torch.from_numpy(rows).cuda()].cpu().numpy()
    if mode == tfd.W_FP8_ROW:
        oc, os_ = quant_fp8_row(wr)
        s_gpu = scales[torch.from_numpy(rows).cuda()].cpu().numpy()
        assert np.array_equal(s_gpu.view(np.uint32), os_.view(np.uint32))
    else:
        oc, os_ = quant_fp8_block32(wr)
        s_gpu = scales[torch.from_numpy(blocks).cuda()].cpu().numpy()
        assert np.array_equal(s_gpu, os_)
    assert np.array_equal(c_gpu, oc)


def test_block32_interleaved_codes_and_relayout():
    """Mode W_FP8_BLOCK32_IL: the plain block-32 codes in the interleaved layout, same scales; the
    relayout converts either way."""
    need_gpu()
    from oracle.quant import block32_interleave
    w = inputs.normal_bf16((256, 4096 + 64), 0.02, 995)
    wd = w.cuda()
    plain, sp = tfd.tfd_quant_fp8(wd, tfd.W_FP8_BLOCK32)
    il, si = tfd.tfd_quant_fp8(wd, tfd.W_FP8_BLOCK32_IL)
    to_il = tfd.tfd_fp8_block32_relayout(plain, True)
    back = tfd.tfd_fp8_block32_relayout(il, False)
    torch.cuda.synchronize()
    oc, os_ = quant_fp8_block32(w.float().numpy())
    assert np.array_equal(plain.cpu().numpy(), oc) and np.array_equal(sp.cpu().numpy(), os_)
    assert np.array_equal(il.cpu().numpy(), block32_interleave(oc))
    assert np.array_equal(si.cpu().numpy(), os_)
    assert torch.equal(to_il, il) and torch.equal(back, plain)
    with pytest.raises(tfd.TfdError):
        tfd.tfd_quant_fp8(inputs.normal_bf16((64, 96), 0.02, 996).cuda(), tfd.W_FP8_BLOCK32_IL)
