"""GPU checks of the expert kernel's building blocks against host-computed expectations:
the hardware E2M1/E4M3 conversions (lane order and values), the TMA 64-byte swizzle
layout, and one tcgen05 MMA with its A operand in tensor memory."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from routed_moe_decode_gb300 import _lib
    lib = _lib.lib()
    lib.moe_selftest_decode.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.moe_selftest_tma.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_void_p, ctypes.c_void_p]
    lib.moe_selftest_mma.argtypes = [ctypes.c_void_p] * 4
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_decode_conversions_match_oracle(L):
    # every byte value in every byte position of a word
    b = np.arange(256, dtype=np.uint32)
    words = (b | (((b + 1) & 255) << 8) | (((b + 7) & 255) << 16) | (((b + 101) & 255) << 24)).astype(np.uint32)
    pairs = np.array([(x | (((x * 37 + 11) & 255) << 8)) for x in range(256)], dtype=np.uint32)
    # keep the E4M3 NaN codes out: they are outside the weight contract
    nan_codes = (0x7F, 0xFF)
    keep = np.array([(p & 255) not in nan_codes and ((p >> 8) & 255) not in nan_codes for p in pairs])
    pairs = pairs[keep]
    dw = torch.from_numpy(words.view(np.int32)).cuda()
    dp = torch.from_numpy(pairs.view(np.int32)).cuda()
    out = torch.zeros(4 * len(words), dtype=torch.int32, device="cuda")
    sout = torch.zeros(len(pairs), dtype=torch.int32, device="cuda")
    assert L.moe_selftest_decode(_p(dw), len(words), _p(out), _p(dp), len(pairs), _p(sout), _s()) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32).view(np.float16).astype(np.float32).reshape(len(words), 8)
    e2m1 = np.array([O.e2m1_value(i) for i in range(16)], np.float32)
    for w_i, w in enumerate(words):
        expect = [e2m1[(int(w) >> (4 * q)) & 15] for q in range(8)]  # element q = nibble q
        np.testing.assert_array_equal(got[w_i], expect)
    sg = sout.cpu().numpy().view(np.uint32).view(np.float16).astype(np.float32).reshape(len(pairs), 2)
    for i, p in enumerate(pairs):
        assert sg[i, 0] == O.e4m3_value(int(p) & 255) and sg[i, 1] == O.e4m3_value((int(p) >> 8) & 255)


def test_tma_box_swizzle_layout(L):
    rng = np.random.default_rng(0)
    rows, row_bytes = 192, 256
    src = rng.integers(0, 256, size=(rows, row_bytes), dtype=np.uint8)
    dsrc = torch.from_numpy(src).cuda()
    out = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    x, y = 128, 64
    assert L.moe_selftest_tma(_p(dsrc), rows, row_bytes, x, y, _p(out), _s()) == 0
    torch.cuda.synchronize()
    img = out.cpu().numpy().reshape(64, 64)
    for r in range(64):
        for c in range(4):  # 16-byte chunk c of row r lands at chunk c ^ ((r >> 1) & 3)
            pos = c ^ ((r >> 1) & 3)
            np.testing.assert_array_equal(img[r, pos * 16:(pos + 1) * 16], src[y + r, x + c * 16:x + (c + 1) * 16])


def test_tcgen05_mma_a_in_tensor_memory(L):
    rng = np.random.default_rng(1)
    # small integers keep every product and sum exact in FP16 inputs / FP32 accumulation
    A = rng.integers(-4, 5, size=(128, 128)).astype(np.float16)
    B = rng.integers(-4, 5, size=(16, 128)).astype(np.float16)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    D = torch.full((128, 16), float("nan"), dtype=torch.float32, device="cuda")
    assert L.moe_selftest_mma(_p(dA), _p(dB), _p(D), _s()) == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(D.cpu().numpy(), A.astype(np.float32) @ B.astype(np.float32).T)
