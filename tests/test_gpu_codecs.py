"""GPU codec and input-generator checks.

The device bf16 -> e4m3 conversion used by the summaries is compared with the oracle's
(pinned) codec over every bf16 bit pattern; the seeded generator draws bit-identical
tensors on the CPU and the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s5():
    import block_sparse_attention_step5_gb300 as s5
    s5.build()
    s5.load()
    return s5


def test_e4m3_conversion_every_bf16_pattern(s5):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).cuda()
    out = torch.empty(65536, dtype=torch.uint8, device="cuda")
    s5.step5_convert_bf16_to_e4m3(x, out)
    got = out.cpu().numpy()
    ref = oracle.bf16_codes_to_e4m3_codes(codes)
    vals = oracle.bf16_values(codes)
    finite = np.isfinite(vals)
    assert np.array_equal(got[finite], ref[finite])
    nan = np.isnan(vals)
    assert np.all((got[nan] & 0x7F) == 0x7F)


def test_generator_identical_on_cpu_and_gpu():
    for stream, scale in ((S.S_K, 1.0), (S.S_IQ, 4.0)):
        a = S.normal_bf16((3, 5, 1000), 17, stream, scale=scale, device="cpu")
        b = S.normal_bf16((3, 5, 1000), 17, stream, scale=scale, device="cuda").cpu()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    u = S.uniform_f32((777,), 41, S.S_W, device="cpu")
    v = S.uniform_f32((777,), 41, S.S_W, device="cuda").cpu()
    assert torch.equal(u, v)
    rows = np.array([3, 17, 4000], dtype=np.int64)
    full = S.normal_bf16((5000, 128), 17, S.S_V, device="cuda").cpu()
    part = S.normal_bf16_rows((5000, 128), rows, 17, S.S_V)
    assert np.array_equal(part[rows], S.codes16(full)[rows])
