"""GPU parity of moe_nvfp4_split (activation rows -> R NVFP4 terms) against the oracle's quantiser."""
import numpy as np
import pytest
import torch

from oracle import formats, nvfp4_split as S
from serving_router_top_gb300 import inputs as I
from serving_router_top_gb300 import moe
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def run_split(src: torch.Tensor, fp32: bool, K: int, R: int):
    rows = src.shape[0]
    codes = torch.zeros((rows * R, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((rows * R, K // 16), dtype=torch.uint8, device="cuda")
    gs = torch.zeros(rows * R, dtype=torch.float32, device="cuda")
    moe.moe_nvfp4_split(src, fp32, rows, K, src.shape[1], R, codes, scales, gs)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy(), gs.cpu().numpy()


def decoded_terms(codes, scales, gs, rows, K, R):
    vals = formats.e2m1_value(formats.unpack_codes(codes))            # [rows*R, K]
    sc = formats.e4m3_value(scales)                                    # [rows*R, K/16]
    t = (vals.reshape(rows * R, K // 16, 16) * sc[:, :, None]).reshape(rows * R, K) * gs[:, None]
    return t.reshape(rows, R, K)


@pytest.mark.parametrize("K", [64, 512, 2048, 4096])
def test_split_bf16_rows_bit_exact(K):
    """bf16 rows (N(0,1), a zero row, rows scaled by 2^-40 and 2^40, rows with a single large
    value): every term's code values, scale bytes and global scales equal the oracle's."""
    R = 4
    g = np.random.default_rng(K)
    x = (g.standard_normal((20, K))).astype(np.float32)
    x[1] = 0.0
    x[2] *= 2.0 ** -40
    x[3] *= 2.0 ** 40
    x[4] = 0.0
    x[4, 7] = 3.0e5
    bits = I.round_f32_to_bf16_bits(x)
    src = torch.from_numpy(bits.view(np.int16)).cuda()
    codes, scales, gs = run_split(src, False, K, R)
    v = formats.bf16_value(bits)
    for i in range(v.shape[0]):
        rest = v[i].copy()
        for r in range(R):
            c, sb, G = S.encode_nvfp4(rest)
            row = i * R + r
            assert gs[row] == np.float32(G), (i, r)
            assert np.array_equal(scales[row], sb), (i, r)
            got = formats.e2m1_value(formats.unpack_codes(codes[row]))
            assert np.array_equal(got, c), (i, r)   # values: +0 and -0 codes compare equal
            rest = rest - (c.reshape(-1, 16) * formats.e4m3_value(sb)[:, None] * G).reshape(-1)


def test_split_fp32_rows_approximate():
    """fp32 rows (the intermediate h): the first term equals the oracle's; the four terms sum to
    within 2^-9 of each row's largest value (the residual is rounded in fp32)."""
    K, R = 512, 4
    g = np.random.default_rng(9)
    h = (g.standard_normal((64, K)) * np.exp(g.uniform(-5, 5, size=(64, 1)))).astype(np.float32)
    src = torch.from_numpy(h).cuda()
    codes, scales, gs = run_split(src, True, K, R)
    t = decoded_terms(codes, scales, gs, 64, K, R)
    for i in range(64):
        c, sb, G = S.encode_nvfp4(h[i].astype(np.float64))
        assert np.array_equal(scales[i * R], sb) and gs[i * R] == np.float32(G)
        err = np.abs(t[i].sum(axis=0) - h[i]).max()
        assert err <= 2.0 ** -9 * np.abs(h[i]).max(), i


def test_split_rejects_bad_arguments():
    x = torch.zeros((4, 512), dtype=torch.int16, device="cuda")
    out = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    g = torch.zeros(64, dtype=torch.float32, device="cuda")
    for K, ld, R in ((500, 512, 4), (512, 256, 4), (512, 512, 0), (512, 512, 9), (8192, 8192, 1)):
        with pytest.raises(moe.MoeError):
            moe.moe_nvfp4_split(x, False, 4, K, ld, R, out, out, g)
