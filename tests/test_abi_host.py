"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/wqgb300.h declares, and refuses bad arguments with the
documented status codes before touching the GPU."""
import ctypes

import pytest

import oracle

wq = pytest.importorskip("weight_only_bit_group_gb300")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__

    __graft_entry__.build()
    return wq.lib()


def test_exports_every_declared_symbol(L):
    names = wq.header_symbols()
    assert len(names) >= 14
    for name in names:
        assert hasattr(L, name), name


def test_status_strings(L):
    for s in range(9):
        assert L.wq_status_string(s)
    assert b"sm_103a" in L.wq_version()


def test_packed_bytes_matches_oracle(L):
    for numel in (0, 1, 7, 8, 63, 64, 1000, 218103808):
        for nbits in range(2, 8):
            assert L.uintx_packed_bytes(numel, nbits) == oracle.uintx_packed_bytes(numel, nbits)
    assert L.uintx_packed_bytes(10, 9) == -1


def test_workspace_sizes(L):
    assert L.wq_workspace_bytes(wq.WQ_OP_GPTQ_QUANTIZE, 4096, 4096, 128) >= 4096 * 16
    assert L.wq_workspace_bytes(wq.WQ_OP_QUANT_SNR, 1, 1, 0) > 0
    awq = L.wq_workspace_bytes(wq.WQ_OP_AWQ_SEARCH, 34816, 5120, 11)
    assert awq >= 2 * 11 * 5120 * 4 + 5120 * 4
    assert L.wq_workspace_bytes(99, 1, 1, 0) == 0


def p(v):
    return ctypes.c_void_p(v)


BAD = p(0x1000)       # never dereferenced: every call below fails its checks first
MIS = p(0x1002)       # misaligned


def test_argument_errors_return_codes(L):
    # shapes
    assert L.mxfp4_quantize(BAD, 4, 48, 0, BAD, BAD, None) == 2
    assert L.mxfp4_quantize(BAD, -1, 64, 0, BAD, BAD, None) == 2
    assert L.gptq_quantize_sym(BAD, 12, 256, 128, BAD, BAD, BAD, BAD, None, None, 0, None) == 2
    assert L.gptq_quantize_asym(BAD, 8, 200, 128, BAD, BAD, BAD, BAD, None, None, 0, None) == 2
    assert L.uintx_quantize(BAD, 4, 100, 4, 64, BAD, BAD, BAD, None) == 2
    # unsupported values (uint8 is refused as the page's can_quantize does)
    assert L.uintx_quantize(BAD, 4, 64, 8, 64, BAD, BAD, BAD, None) == 5
    assert L.uintx_quantize(BAD, 4, 64, 1, 64, BAD, BAD, BAD, None) == 5
    assert L.gptq_quantize_sym(BAD, 8, 256, 96, BAD, BAD, BAD, BAD, None, None, 0, None) == 5
    assert L.mxfp4_quantize(BAD, 4, 64, 7, BAD, BAD, None) == 5
    # dtypes / layouts
    assert L.mxfp4_dequantize(BAD, BAD, 4, 64, 5, BAD, None) == 3
    assert L.quant_snr(BAD, BAD, 9, 0, 4, 64, BAD, BAD, BAD, 1 << 20, None) == 3
    assert L.gptq_dequantize(BAD, BAD, BAD, 8, 128, 128, 1, 0, 7, BAD, None) == 5
    # null pointers
    assert L.mxfp4_quantize(None, 4, 64, 0, BAD, BAD, None) == 1
    assert L.gptq_quantize_sym(BAD, 8, 128, 128, None, BAD, BAD, BAD, None, None, 0, None) == 1
    assert L.gptq_quantize_sym(BAD, 8, 128, 128, BAD, BAD, BAD, BAD, BAD, None, 0, None) == 1
    # misalignment
    assert L.mxfp4_quantize(MIS, 4, 64, 0, BAD, BAD, None) == 4
    assert L.uintx_quantize(BAD, 4, 64, 4, 64, MIS, BAD, BAD, None) == 4
    # workspace too small
    assert L.gptq_quantize_asym(BAD, 8, 128, 128, BAD, BAD, BAD, BAD, BAD, BAD, 16, None) == 6
    assert L.quant_snr(BAD, BAD, 0, 0, 4, 64, BAD, BAD, BAD, 16, None) == 6
    al = (ctypes.c_float * 2)(0.0, 1.0)
    assert L.awq_search(BAD, 64, 64, BAD, al, 2, 16, 0, BAD, BAD, BAD, BAD, BAD, 16, None) == 6
    assert L.awq_search(BAD, 64, 64, BAD, al, 17, 16, 0, BAD, BAD, BAD, BAD, BAD, 1 << 30, None) == 5


def test_awq_fold_argument_errors(L):
    assert L.awq_fold(BAD, 4, 60, BAD, 0, 0, BAD, None) == 2     # k % 8 != 0
    assert L.awq_fold(BAD, -1, 64, BAD, 0, 0, BAD, None) == 2
    assert L.awq_fold(BAD, 4, 64, BAD, 2, 0, BAD, None) == 5     # no such axis
    assert L.awq_fold(BAD, 4, 64, BAD, 0, 3, BAD, None) == 5     # no such op
    assert L.awq_fold(BAD, 4, 64, None, 0, 0, BAD, None) == 1
    assert L.awq_fold(MIS, 4, 64, BAD, 0, 0, BAD, None) == 4
    assert L.awq_fold(BAD, 4, 64, p(0x1004), 0, 0, BAD, None) == 4   # column scales need 16 B
    assert L.awq_fold(None, 0, 64, None, 1, 1, None, None) == 0      # empty: nothing launched


def test_gptq_linear_argument_errors(L):
    ws = L.gptq_linear_workspace_bytes(1, 4096)
    assert ws >= 64 * 4096 * 4 and L.gptq_linear_workspace_bytes(9, 4096) == 0
    assert L.gptq_linear(BAD, 9, BAD, BAD, BAD, 64, 128, 128, 1, 0, BAD, BAD, 1 << 30, None) == 5
    assert L.gptq_linear(BAD, 1, BAD, BAD, BAD, 64, 100, 128, 1, 0, BAD, BAD, 1 << 30, None) == 2
    assert L.gptq_linear(BAD, 1, BAD, BAD, BAD, 64, 128, 96, 1, 0, BAD, BAD, 1 << 30, None) == 5
    assert L.gptq_linear(BAD, 1, BAD, BAD, BAD, 64, 128, 128, 1, 7, BAD, BAD, 1 << 30, None) == 3
    assert L.gptq_linear(BAD, 1, BAD, None, BAD, 64, 128, 128, 0, 0, BAD, BAD, 1 << 30, None) == 1
    assert L.gptq_linear(BAD, 1, BAD, BAD, BAD, 64, 128, 128, 1, 0, BAD, BAD, 16, None) == 6
    assert L.gptq_linear(MIS, 1, BAD, BAD, BAD, 64, 128, 128, 1, 0, BAD, BAD, 1 << 30, None) == 4
    assert L.gptq_linear(None, 0, None, None, None, 64, 128, 128, 1, 0, None, None, 0, None) == 0


def test_gptq_gemm_argument_errors(L):
    assert L.gptq_gemm(BAD, 16, BAD, BAD, BAD, 64, 128, 96, 1, 0, BAD, None) == 5      # group
    assert L.gptq_gemm(BAD, 16, BAD, BAD, BAD, 64, 100, 128, 1, 0, BAD, None) == 2     # k % group
    assert L.gptq_gemm(BAD, 16, BAD, BAD, BAD, 60, 128, 128, 1, 0, BAD, None) == 2     # n % 8
    assert L.gptq_gemm(BAD, -1, BAD, BAD, BAD, 64, 128, 128, 1, 0, BAD, None) == 2
    assert L.gptq_gemm(BAD, 16, BAD, BAD, BAD, 64, 128, 128, 1, 7, BAD, None) == 3
    assert L.gptq_gemm(BAD, 16, BAD, None, BAD, 64, 128, 128, 0, 0, BAD, None) == 1    # asym needs qzeros
    assert L.gptq_gemm(BAD, 16, BAD, BAD, BAD, 64, 128, 128, 1, 0, None, None) == 1
    assert L.gptq_gemm(MIS, 16, BAD, BAD, BAD, 64, 128, 128, 1, 0, BAD, None) == 4
    assert L.gptq_gemm(BAD, 16, MIS, BAD, BAD, 64, 128, 128, 1, 0, BAD, None) == 4
    assert L.gptq_gemm(None, 0, None, None, None, 64, 128, 128, 1, 0, None, None) == 0


def test_uintx_gemm_argument_errors(L):
    assert L.uintx_gemm(BAD, 16, BAD, BAD, BAD, 64, 128, 8, 64, 0, BAD, None) == 5     # nbits 8
    assert L.uintx_gemm(BAD, 16, BAD, BAD, BAD, 64, 128, 1, 64, 0, BAD, None) == 5     # nbits 1
    assert L.uintx_gemm(BAD, 16, BAD, BAD, BAD, 64, 128, 4, 48, 0, BAD, None) == 5     # group
    assert L.uintx_gemm(BAD, 16, BAD, BAD, BAD, 64, 96, 4, 32, 0, BAD, None) == 5      # k % 64
    assert L.uintx_gemm(BAD, 16, BAD, BAD, BAD, 64, 192, 4, 128, 0, BAD, None) == 2    # k % group
    assert L.uintx_gemm(BAD, 16, BAD, BAD, BAD, 64, 128, 4, 64, 7, BAD, None) == 3
    assert L.uintx_gemm(BAD, 16, BAD, None, BAD, 64, 128, 4, 64, 0, BAD, None) == 1
    assert L.uintx_gemm(BAD, 16, MIS, BAD, BAD, 64, 128, 4, 64, 0, BAD, None) == 4
    assert L.uintx_gemm(None, 0, None, None, None, 64, 128, 4, 64, 0, None, None) == 0


def test_wide_quantize_argument_errors(L):
    ws = 1 << 20
    # dtype 7 is no weight type; uint8 outputs etc. are not checked before the dtype
    assert L.gptq_quantize_ex(BAD, 7, 64, 128, 128, 1, BAD, BAD, BAD, BAD, None, None, 0, None) == 3
    assert L.gptq_quantize_ex(BAD, 0, 64, 128, 96, 1, BAD, BAD, BAD, BAD, None, None, 0, None) == 5
    assert L.gptq_quantize_ex(BAD, 2, 60, 128, 128, 1, BAD, BAD, BAD, BAD, None, None, 0, None) == 2
    assert L.gptq_quantize_ex(BAD, 0, 64, 128, 128, 1, None, BAD, BAD, BAD, None, None, 0, None) == 1
    assert L.gptq_quantize_ex(BAD, 0, 64, 128, 128, 0, BAD, BAD, BAD, BAD, BAD, BAD, 16, None) == 6
    assert L.gptq_quantize_ex(MIS, 2, 64, 128, 128, 1, BAD, BAD, BAD, BAD, None, None, 0, None) == 4
    assert L.gptq_quantize_ex(None, 0, 0, 128, 128, 1, None, None, None, None, None, None, 0, None) == 0
    assert L.mxfp4_quantize_ex(BAD, 7, 64, 64, 0, BAD, BAD, None) == 3
    assert L.mxfp4_quantize_ex(BAD, 0, 64, 48, 0, BAD, BAD, None) == 2
    assert L.mxfp4_quantize_ex(BAD, 2, 64, 64, 5, BAD, BAD, None) == 5
    assert L.mxfp4_quantize_ex(MIS, 0, 64, 64, 0, BAD, BAD, None) == 4
    assert L.mxfp4_quantize_ex(None, 2, 0, 64, 0, None, None, None) == 0
    assert ws  # (the SNR workspace size is the bf16 path's)
    assert L.uintx_quantize_ex(BAD, 7, 8, 64, 4, 64, BAD, BAD, BAD, None) == 3
    assert L.uintx_quantize_ex(BAD, 0, 8, 64, 8, 64, BAD, BAD, BAD, None) == 5     # nbits 8
    assert L.uintx_quantize_ex(BAD, 2, 8, 64, 4, 12, BAD, BAD, BAD, None) == 2     # group % 8
    assert L.uintx_quantize_ex(BAD, 0, 8, 64, 4, 48, BAD, BAD, BAD, None) == 2     # k % group
    assert L.uintx_quantize_ex(BAD, 0, 8, 64, 4, 64, None, BAD, BAD, None) == 1
    assert L.uintx_quantize_ex(MIS, 0, 8, 64, 4, 64, BAD, BAD, BAD, None) == 4     # fp32 needs 4-byte
    assert L.uintx_quantize_ex(None, 2, 0, 64, 4, 64, None, None, None, None) == 0
    assert L.uintx_dequantize_ex(BAD, BAD, 7, BAD, 8, 64, 4, 64, BAD, None) == 3
    assert L.uintx_dequantize_ex(BAD, BAD, 2, BAD, 8, 64, 1, 64, BAD, None) == 5
    assert L.uintx_dequantize_ex(BAD, BAD, 0, BAD, 8, 64, 4, 64, None, None) == 1


def test_mxfp4_linear_argument_errors(L):
    assert L.mxfp4_linear(BAD, 1, BAD, BAD, 64, 48, 0, BAD, None) == 2     # k % 32 != 0
    assert L.mxfp4_linear(BAD, 9, BAD, BAD, 64, 64, 0, BAD, None) == 5     # m > 8
    assert L.mxfp4_linear(BAD, 1, BAD, BAD, 64, 64, 5, BAD, None) == 3
    assert L.mxfp4_linear(BAD, 1, None, BAD, 64, 64, 0, BAD, None) == 1
    assert L.mxfp4_linear(MIS, 1, BAD, BAD, 64, 64, 0, BAD, None) == 4
    assert L.mxfp4_linear(None, 0, None, None, 64, 64, 0, None, None) == 0


def test_empty_inputs_are_ok_without_gpu(L):
    assert L.mxfp4_quantize(None, 0, 64, 0, None, None, None) == 0
    assert L.uintx_dequantize(None, None, None, 3, 0, 4, 64, 1, None, None) == 0
    assert L.gptq_dequantize(None, None, None, 0, 128, 128, 1, 0, 0, None, None) == 0


def test_consumers_refuse_non_bf16_operands():
    import torch

    x16 = torch.zeros(2, 64, dtype=torch.float16)
    for call in (lambda: wq.gptq_gemm(x16, None, None, None, 64, 64),
                 lambda: wq.gptq_linear(x16, None, None, None, 64, 64),
                 lambda: wq.mxfp4_linear(x16, torch.zeros(64, 32, dtype=torch.uint8), None),
                 lambda: wq.uintx_gemm(x16, None, None, None, 64, 64, 4)):
        with pytest.raises(TypeError):
            call()
    with pytest.raises(TypeError):
        wq.uintx_gemm(torch.zeros(2, 64, dtype=torch.bfloat16), None,
                      torch.zeros(64, 1, dtype=torch.float16), None, 64, 64, 4)


# ------------------------------------------------------------------ binding argument checks
# The kernels size every read and write from the shape arguments, so the binding
# checks each tensor before the call.  These run on CPU tensors: every case must
# raise before the library is reached (a CPU tensor that passed every check would
# still be refused as not on a CUDA device).
def _cpu(shape, dtype):
    import torch

    return torch.zeros(shape, dtype=dtype)


def test_binding_refuses_output_dtypes_the_library_does_not_write():
    import torch

    qw, qz, sc = _cpu((16, 64), torch.int32), _cpu((1, 8), torch.int32), _cpu((1, 64), torch.float16)
    with pytest.raises(TypeError):  # float16 output would be written as binary32
        wq.gptq_dequantize(qw, qz, sc, 64, 128, 128, False, out_dtype=torch.float16)
    with pytest.raises(TypeError):
        wq.mxfp4_dequantize(_cpu((4, 32), torch.uint8), _cpu((4, 2), torch.uint8), out_dtype=torch.float16)
    with pytest.raises(TypeError):
        wq.uintx_dequantize(_cpu((256,), torch.uint8), _cpu((4, 2), torch.bfloat16), _cpu((4, 2), torch.uint8),
                            4, 128, 4, 64, out_dtype=torch.float64)
    x = _cpu((1, 128), torch.bfloat16)
    for call in (lambda: wq.gptq_linear(x, qw, qz, sc, 64, 128, 128, False, out_dtype=torch.float16),
                 lambda: wq.gptq_gemm(x, qw, qz, sc, 64, 128, 128, False, out_dtype=torch.float16),
                 lambda: wq.mxfp4_linear(x, _cpu((4, 64), torch.uint8), _cpu((4, 4), torch.uint8),
                                         out_dtype=torch.float16)):
        with pytest.raises(TypeError):
            call()
    # quant_snr: an fp16 deq would be read as binary32
    with pytest.raises(TypeError):
        wq.quant_snr(_cpu((4, 64), torch.bfloat16), _cpu((4, 64), torch.float16))


def test_binding_checks_caller_outputs():
    import torch

    qw, qz, sc = _cpu((16, 64), torch.int32), _cpu((1, 8), torch.int32), _cpu((1, 64), torch.float16)
    # out whose dtype differs from out_dtype: the kernel would write 4 bytes per 2-byte element
    with pytest.raises(TypeError, match="out"):
        wq.gptq_dequantize(qw, qz, sc, 64, 128, 128, False, torch.float32, out=_cpu((64, 128), torch.bfloat16))
    with pytest.raises(TypeError, match="out"):
        wq.mxfp4_dequantize(_cpu((4, 32), torch.uint8), _cpu((4, 2), torch.uint8),
                            out=_cpu((4, 64), torch.bfloat16))
    # too few elements
    with pytest.raises(ValueError, match="out"):
        wq.gptq_dequantize(qw, qz, sc, 64, 128, 128, False, torch.float32, out=_cpu((64, 127), torch.float32))
    with pytest.raises(ValueError, match="packed"):
        wq.mxfp4_quantize(_cpu((4, 64), torch.bfloat16), packed=_cpu((4, 31), torch.uint8))
    with pytest.raises(ValueError, match="scales"):
        wq.gptq_quantize_asym(_cpu((64, 128), torch.bfloat16), 128, scales=_cpu((1, 63), torch.float16))
    with pytest.raises(ValueError, match="zp"):
        wq.uintx_quantize(_cpu((4, 128), torch.bfloat16), 4, 64, zp=_cpu((4, 1), torch.uint8))
    # not contiguous
    with pytest.raises(ValueError, match="contiguous"):
        wq.gptq_dequantize(qw, qz, sc, 64, 128, 128, False, torch.float32,
                           out=_cpu((128, 64), torch.float32).t())
    # a workspace that is too small or of the wrong type
    with pytest.raises(ValueError, match="ws"):
        wq.quant_snr(_cpu((4, 64), torch.bfloat16), _cpu((4, 64), torch.float32), ws=_cpu((16,), torch.uint8))
    with pytest.raises(TypeError, match="ws"):
        wq.gptq_quantize_sym(_cpu((64, 128), torch.bfloat16), 128, ws=_cpu((1 << 20,), torch.float32))
    # everything consistent: still refused, the tensors are not on a CUDA device
    with pytest.raises(ValueError, match="CUDA"):
        wq.gptq_dequantize(qw, qz, sc, 64, 128, 128, False, torch.float32, out=_cpu((64, 128), torch.float32))


def test_binding_checks_inputs():
    import torch

    # the stored GPTQ tensors must match n, k, group
    with pytest.raises(ValueError, match="qweight"):
        wq.gptq_dequantize(_cpu((15, 64), torch.int32), None, _cpu((1, 64), torch.float16), 64, 128, 128, True)
    with pytest.raises(ValueError, match="qzeros"):  # asym needs its zero points
        wq.gptq_dequantize(_cpu((16, 64), torch.int32), None, _cpu((1, 64), torch.float16), 64, 128, 128, False)
    with pytest.raises(ValueError, match="e8m0"):
        wq.mxfp4_dequantize(_cpu((4, 32), torch.uint8), _cpu((4, 1), torch.uint8))
    with pytest.raises(ValueError, match="packed"):
        wq.uintx_dequantize(_cpu((255,), torch.uint8), _cpu((4, 2), torch.bfloat16), _cpu((4, 2), torch.uint8),
                            4, 128, 4, 64)
    # 16-bit weights other than bf16 would be read as bf16 bit patterns
    a = _cpu((64,), torch.float32)
    for call in (lambda: wq.awq_search(_cpu((4, 64), torch.float16), a, [0.0, 1.0]),
                 lambda: wq.awq_fold(_cpu((4, 64), torch.float16), a),
                 lambda: wq.quant_snr(_cpu((4, 64), torch.float16), _cpu((4, 64), torch.float32)),
                 lambda: wq.gptq_quantize_sym(_cpu((64, 128), torch.int16), 128)):
        with pytest.raises(TypeError):
            call()
    # the activation statistics: binary32, one per column
    with pytest.raises(TypeError, match="a"):
        wq.awq_search(_cpu((4, 64), torch.bfloat16), _cpu((64,), torch.float64), [0.0, 1.0])
    with pytest.raises(ValueError, match="a"):
        wq.awq_search(_cpu((4, 64), torch.bfloat16), _cpu((32,), torch.float32), [0.0, 1.0])
    # fold scales: k entries per column fold, n per row fold
    with pytest.raises(ValueError, match="s"):
        wq.awq_fold(_cpu((4, 64), torch.bfloat16), _cpu((4,), torch.float32), axis=0)
    with pytest.raises(ValueError, match="layout"):
        wq.quant_snr(_cpu((4, 64), torch.bfloat16), _cpu((4, 64), torch.float32), layout="mk")
    # consumers: x must have the weight's k columns
    with pytest.raises(ValueError, match="columns"):
        wq.gptq_gemm(_cpu((2, 96), torch.bfloat16), _cpu((16, 64), torch.int32), None,
                     _cpu((1, 64), torch.float16), 64, 128)
