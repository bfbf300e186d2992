"""Bit-exact MXFP4 decoding on the GPU: every packed byte x every e8m0
scale byte through both device decoders, against the oracle."""
import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from oracle import oracle as ora

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def all_pairs():
    packed = np.tile(np.arange(256, dtype=np.uint8), (256, 1))  # row S holds every byte
    scale = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 512 // 32, axis=1)
    return packed, scale


def gpu_dequant(packed, scale, kind):
    rows, cols = packed.shape[0], packed.shape[1] * 2
    p = torch.from_numpy(packed).cuda()
    s = torch.from_numpy(scale).cuda()
    if kind == 0:
        out = torch.empty((rows, cols), dtype=torch.int16, device="cuda")
    else:
        out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    k3moe.mxfp4_dequant(p, s, rows, cols, out, kind, torch.cuda.current_stream())
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    return o.view(np.uint16) if kind == 0 else o


def test_bf16_tile_decoder_bit_exact_all_bytes_all_scales():
    packed, scale = all_pairs()
    got = gpu_dequant(packed, scale, 0)
    ref = ora.mxfp4_dequant_bf16(packed, scale)
    fin = np.isfinite(ora.bf16_to_float(ref))
    # scale bytes 0..252: every value is exact and must match bit for bit
    assert np.array_equal(got[:253], ref[:253])
    # 253, 254: IEEE overflow to infinity in the same places, same bits elsewhere
    assert np.array_equal(got[253:255], ref[253:255])
    # 255 (NaN scale): NaN everywhere
    assert np.all(np.isnan(ora.bf16_to_float(got[255])))
    assert fin[:253].all()


def test_fp32_decoder_bit_exact_all_bytes_all_scales():
    packed, scale = all_pairs()
    got = gpu_dequant(packed, scale, 1)
    ref = ora.bf16_to_float(ora.mxfp4_dequant_bf16(packed, scale)).astype(np.float32)
    assert np.array_equal(got[:255].view(np.uint32), ref[:255].view(np.uint32))
    assert np.all(np.isnan(got[255]))


def test_decoders_on_random_matrix_with_ragged_rows():
    rng = np.random.default_rng(0)
    rows, cols = 333, 1024
    packed = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    scale = rng.integers(100, 140, (rows, cols // 32), dtype=np.uint8)
    ref = ora.mxfp4_dequant_bf16(packed, scale)
    assert np.array_equal(gpu_dequant(packed, scale, 0), ref)
    assert np.array_equal(gpu_dequant(packed, scale, 1), ora.bf16_to_float(ref).astype(np.float32))


def test_k3_expert_tensor_slice():
    from mxfp4_routed_expert_k3_gb300.dims import K3
    packed = synth.u8_full(11, 6, (256, K3.latent // 2))
    scale = synth.u8_range(11, 7, (256, K3.latent // 32), 118, 124)
    ref = ora.mxfp4_dequant_bf16(packed, scale)
    assert np.array_equal(gpu_dequant(packed, scale, 0), ref)
