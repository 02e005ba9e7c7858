"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point that include/gguf_gb300.h declares, and rejects bad
arguments with the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gguf_gb300.h")


@pytest.fixture(scope="module")
def g():
    from gguf_block_quantized_quantize_gb300 import build

    build.build()
    import gguf_block_quantized_quantize_gb300 as g

    g.load_library()
    return g


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gguf_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(g):
    names = _declared()
    assert "gguf_mul_mat" in names and "gguf_mul_mat_id" in names and "gguf_quantize_q8_1" in names
    lib = ctypes.CDLL(g.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
        assert n in g.SIGNATURES, f"binding lacks {n}"


def test_type_table(g):
    L = g.load_library()
    assert L.gguf_type_block_elems(g.Q4_K) == 256 and L.gguf_type_block_bytes(g.Q4_K) == 144
    assert L.gguf_type_block_elems(g.Q6_K) == 256 and L.gguf_type_block_bytes(g.Q6_K) == 210
    assert L.gguf_type_block_elems(g.Q8_0) == 32 and L.gguf_type_block_bytes(g.Q8_0) == 34
    assert L.gguf_type_block_elems(g.Q8_1) == 32 and L.gguf_type_block_bytes(g.Q8_1) == 36
    assert L.gguf_type_block_elems(g.Q4_0) == 32 and L.gguf_type_block_bytes(g.Q4_0) == 18
    assert L.gguf_type_block_elems(g.Q5_K) == 256 and L.gguf_type_block_bytes(g.Q5_K) == 176
    assert g.gguf_row_size(g.Q4_0, 4128) == 2322 and g.gguf_row_size(g.Q5_K, 2048) == 1408
    assert L.gguf_type_block_elems(g.MXFP4) == 32 and L.gguf_type_block_bytes(g.MXFP4) == 17
    assert g.gguf_row_size(g.MXFP4, 4128) == 2193
    assert g.gguf_row_size(g.Q4_K, 4096) == 2304 and g.gguf_row_size(g.Q6_K, 3072) == 2520
    assert g.gguf_row_size(g.Q4_K, 100) == -1 and L.gguf_type_block_bytes(99) == 0


FAKE = ctypes.c_void_p(0x10000)    # never dereferenced: validation fails first


def _mm(g, **kw):
    a = dict(w=FAKE, wt=g.Q4_K, n=16, k=256, x=FAKE, xt=g.F32, m=4, ldx=256, y=FAKE, yt=g.F32, ldy=16,
             ws=FAKE, ws_bytes=1 << 20)
    a.update(kw)
    L = g.load_library()
    return L.gguf_mul_mat(a["w"], a["wt"], a["n"], a["k"], a["x"], a["xt"], a["m"], a["ldx"], a["y"], a["yt"],
                          a["ldy"], a["ws"], a["ws_bytes"], None)


def test_mul_mat_rejects_bad_arguments(g):
    assert _mm(g, wt=3) == 2                       # Q4_1: unsupported type
    assert _mm(g, xt=g.Q6_K) == 2
    assert _mm(g, yt=g.Q8_0) == 2
    assert _mm(g, k=100) == 3                      # not a multiple of 256
    assert _mm(g, n=-1) == 1
    assert _mm(g, ldy=8) == 1
    assert _mm(g, ldx=128) == 1
    assert _mm(g, w=None) == 1
    assert _mm(g, w=ctypes.c_void_p(0x10008)) == 4  # weight base not 16-byte aligned
    assert _mm(g, ws=None, ws_bytes=0) == 5         # float x needs a q8_1 workspace
    assert _mm(g, ws_bytes=16) == 5
    assert "workspace" in g.load_library().gguf_last_error().decode()
    assert _mm(g, m=0) == 0 and _mm(g, n=0) == 0     # empty products are no-ops


def test_workspace_sizes(g):
    assert g.gguf_mul_mat_ws_size(g.Q4_K, 4096, 4096, g.Q8_1, 8) == 0
    assert g.gguf_mul_mat_ws_size(g.Q4_K, 4096, 4096, g.BF16, 8) >= 8 * 4096 // 32 * 36
    assert g.gguf_mul_mat_ws_size(g.Q4_K, 4096, 4096, g.BF16, 64) >= 64 * 4096 * 2
    # fp32 outputs of the tensor-core path also hold the low fp16 parts
    assert g.gguf_mul_mat_ws_size(g.Q4_K, 4096, 4096, g.BF16, 64, g.F32) >= 2 * 64 * 4096 * 2


def test_other_entry_points_reject_bad_arguments(g):
    L = g.load_library()
    assert L.gguf_quantize_q8_1(FAKE, g.Q8_0, 4, 64, 64, FAKE, None) == 2
    assert L.gguf_quantize_q8_1(FAKE, g.F32, 4, 40, 40, FAKE, None) == 3
    assert L.gguf_quantize_q8_1(FAKE, g.F32, 4, 64, 32, FAKE, None) == 1
    assert L.gguf_dequantize(FAKE, 3, 4, 64, FAKE, g.F32, None) == 2     # Q4_1: not supported
    assert L.gguf_dequantize(FAKE, g.Q6_K, 4, 300, FAKE, g.F32, None) == 3
    assert L.gguf_dequantize(FAKE, g.Q6_K, 4, 256, FAKE, g.Q8_0, None) == 2
    assert L.gguf_get_rows(FAKE, g.Q6_K, 4, 256, None, 3, FAKE, g.F32, None) == 1
    assert L.gguf_debug_block_dots(FAKE, g.F32, 4, 256, FAKE, 1, FAKE, None) == 2
    assert L.gguf_set_option(b"no_such_key", 1) == 1
    assert L.gguf_set_option(b"mmvq_max_m", 8) == 0 and L.gguf_get_option(b"mmvq_max_m") == 8
    assert L.gguf_get_option(b"mmvq_tc") == 1
    assert L.gguf_get_option(b"mmvq_tc_min_m") == 5
    assert L.gguf_set_option(b"mmvq_tc_min_m", 0) != 0 and L.gguf_get_option(b"mmvq_tc_min_m") == 5
    assert L.gguf_get_option(b"moe_vec_max_tokens") == 256
    assert L.gguf_set_option(b"moe_vec_max_tokens", 257) != 0 and L.gguf_get_option(b"moe_vec_max_tokens") == 256
    assert L.gguf_get_option(b"mmvq_tc_max_m") == 16
    assert L.gguf_set_option(b"mmvq_tc_max_m", 64) != 0 and L.gguf_get_option(b"mmvq_tc_max_m") == 16
    assert L.gguf_get_option(b"mmq_stage") == 1 and L.gguf_get_option(b"moe_deterministic") == 1
    assert L.gguf_set_option(b"moe_deterministic", 0) == 0 and L.gguf_get_option(b"moe_deterministic") == 0
    assert L.gguf_set_option(b"moe_deterministic", 1) == 0
    assert L.gguf_get_option(b"moe_down_precise") == 0
    assert L.gguf_get_option(b"moe_gate_up_precise") == 1
    assert L.gguf_set_option(b"moe_gate_up_precise", 0) == 0 and L.gguf_get_option(b"moe_gate_up_precise") == 0
    assert L.gguf_set_option(b"moe_gate_up_precise", 1) == 0
    assert L.gguf_get_option(b"mmq_bn_max") == 256 and L.gguf_get_option(b"mmq_split_k") == 1
    assert L.gguf_get_option(b"mmq_engine") == 0 and L.gguf_set_option(b"mmq_engine", 2) != 0
    assert L.gguf_set_option(b"mmq_engine", 1) == 0 and L.gguf_get_option(b"mmq_engine") == 1
    assert L.gguf_set_option(b"mmq_engine", 0) == 0


def _moe(g, **kw):
    """gguf_mul_mat_id on fake device pointers: only the synchronous argument
    checks run (every call below fails validation before any launch, or has
    no tokens)."""
    a = dict(w=0x10000, wt=g.Q4_K, n_experts=4, expert_stride=256 * 144, n=256, k=256, x=0x20000, xt=g.BF16,
             n_tokens=3, ldx=256, ids=0x30000, top_k=2, route_w=0, mode=g.PLAIN, y=0x40000, yt=g.F32,
             dev_status=0)
    a.update(kw)
    args = g.MoeArgs(a["w"], a["wt"], a["n_experts"], a["expert_stride"], a["n"], a["k"], a["x"], a["xt"],
                     a["n_tokens"], a["ldx"], a["ids"], a["top_k"], a["route_w"], a["mode"], a["y"], a["yt"],
                     a["dev_status"])
    L = g.load_library()
    return L.gguf_mul_mat_id(ctypes.byref(args), FAKE, 0, None)


def test_mul_mat_id_modes_and_types(g):
    assert g.GATE_UP_SWIGLU == 0 and g.DOWN_WEIGHTED_SUM == 1 and g.PLAIN == 2
    assert _moe(g, mode=3) == 1                       # unknown mode
    assert _moe(g, yt=g.Q8_1) == 2                    # PLAIN rows are float
    assert _moe(g, mode=g.DOWN_WEIGHTED_SUM, yt=g.Q8_1) == 2
    assert _moe(g, wt=3) == 2                         # Q4_1: not a supported bank type
    assert _moe(g, k=100) == 3                        # not a multiple of the Q4_K block
    assert _moe(g, expert_stride=256 * 144 - 16) == 1  # stride below n * row_size
    assert _moe(g, n_tokens=0) == 0                   # no tokens: nothing to do
    # the remaining valid PLAIN call fails only on the (absent) workspace
    assert _moe(g) == 5 and "workspace" in g.load_library().gguf_last_error().decode()
    for wt, k in ((g.Q4_0, 96), (g.MXFP4, 96), (g.Q5_K, 256), (g.Q8_0, 64)):
        stride = -(-256 * g.gguf_row_size(wt, k) // 16) * 16
        assert _moe(g, wt=wt, k=k, ldx=k, expert_stride=stride) == 5, wt


def test_noalloc_argument_checks(g):
    L = g.load_library()

    def na(**kw):
        a = dict(w=FAKE, wt=g.Q4_K, n=16, k=256, x=FAKE, xt=g.BF16, m=4, ldx=256, y=FAKE, yt=g.BF16, ldy=16)
        a.update(kw)
        return L.gguf_mul_mat_noalloc(a["w"], a["wt"], a["n"], a["k"], a["x"], a["xt"], a["m"], a["ldx"], a["y"],
                                      a["yt"], a["ldy"], None)
    assert na(k=0, ldx=0) == 3                 # k == 0 with rows to compute: as gguf_mul_mat
    assert _mm(g, k=0, ldx=0) == 3
    assert na(m=0) == 0 and na(n=0) == 0       # empty products are no-ops
    assert na(m=9) == 5 and na(k=16640, ldx=16640) == 5   # beyond the fixed scratch
    assert na(xt=g.Q8_1) == 2
    assert na(ldx=128) == 1


def test_binding_rejects_strided_rows(g):
    import torch
    # checked before any pointer reaches the library (CPU tensors, nothing launched)
    xt = torch.zeros(256, 4, dtype=torch.bfloat16).t()          # [4, 256] with stride(1) == 4
    w = torch.zeros(16 * 144, dtype=torch.uint8)
    for fn in (lambda: g.gguf_mul_mat(w, g.Q4_K, 16, 256, xt),
               lambda: g.gguf_mul_mat_noalloc(w, g.Q4_K, 16, 256, xt),
               lambda: g.gguf_mul_mat_segments(g.Q4_K, 256, xt, [(w, 16, torch.zeros(4, 16, dtype=torch.bfloat16))])):
        with pytest.raises(ValueError):
            fn()
    # q8_1 rows with a gap between them
    xq = torch.zeros(4, 2 * 288, dtype=torch.uint8)[:, :288]
    with pytest.raises(ValueError):
        g.gguf_mul_mat(w, g.Q4_K, 16, 256, xq, xt=g.Q8_1)


def test_device_error_query_arguments(g):
    L = g.load_library()
    # null flags: refused before any CUDA call
    assert L.gguf_device_errors(None, 1, None) == 1
    assert L.gguf_device_errors_async(None, 1, None) == 1
    assert L.gguf_device_errors_async(ctypes.c_void_p(0x10002), 1, None) == 4
    assert g._STATUS[7] == "DEVICE"


def test_mul_mat_batch_argument_checks(g):
    L = g.load_library()
    seg = g.Segment(FAKE, 16, FAKE, 16)
    segs = (g.Segment * 1)(seg)
    def job(m, nseg=1, xq=0x20000):
        return g.MmJob(segs, nseg, ctypes.c_void_p(xq), m)
    def run(jobs, wt=None, k=256, yt=None):
        arr = (g.MmJob * max(len(jobs), 1))(*jobs) if jobs else None
        return L.gguf_mul_mat_batch(g.Q4_K if wt is None else wt, k, arr, len(jobs), g.BF16 if yt is None else yt, None)
    assert run([]) == 0                                    # no jobs: nothing to do
    assert run([job(4)] * 9) == 1                          # more than GGUF_MAX_BATCH_JOBS
    assert run([job(4, nseg=0)]) == 1
    assert run([job(4)], wt=3) == 2                        # Q4_1: unsupported
    assert run([job(4)], yt=g.Q8_0) == 2
    assert run([job(4)], k=100) == 3
    assert run([job(4), job(64)]) == 1                     # m = 64 is not decode-sized
    assert "decode-sized" in L.gguf_last_error().decode()
    assert run([job(4, xq=0x20002)]) == 4                  # q8_1 rows must be 4-byte aligned
    assert run([job(0)]) == 0                              # empty jobs are skipped


def test_copy_argument_checks(g):
    L = g.load_library()
    assert L.gguf_copy_async(None, None, 0, None) == 0          # nothing to copy
    assert L.gguf_copy_async(FAKE, FAKE, -1, None) == 1         # negative size
    assert L.gguf_copy_async(None, FAKE, 16, None) == 1         # null pointer
    # pageable host memory is not device-accessible: refused before any launch
    buf = ctypes.create_string_buffer(64)
    assert L.gguf_copy_async(ctypes.addressof(buf), ctypes.addressof(buf) + 32, 16, None) == 1
    assert "device, managed or pinned" in L.gguf_last_error().decode()
    # the binding refuses pageable and non-contiguous tensors and size mismatches
    with pytest.raises(ValueError):
        g.gguf_copy(torch.zeros(16, dtype=torch.uint8), torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError):
        g.gguf_copy(torch.zeros(4, 4)[:, :2], torch.zeros(8))


def test_mul_mat_batch_typed_argument_checks(g):
    L = g.load_library()
    seg = g.Segment(FAKE, 16, FAKE, 16)
    segs = (g.Segment * 1)(seg)
    def job(wt, k, m, xq=0x20000):
        return g.MmJobTyped(wt, k, segs, 1, ctypes.c_void_p(xq), m)
    def run(jobs, yt=None):
        arr = (g.MmJobTyped * max(len(jobs), 1))(*jobs) if jobs else None
        return L.gguf_mul_mat_batch_typed(arr, len(jobs), g.BF16 if yt is None else yt, None)
    assert run([]) == 0
    assert run([job(g.Q4_K, 256, 4)] * 9) == 1              # more than GGUF_MAX_BATCH_JOBS
    assert run([job(g.Q4_K, 256, 4), job(3, 256, 4)]) == 2  # the second job's type (Q4_1) is unsupported
    assert "job 1" in L.gguf_last_error().decode()
    assert run([job(g.Q4_K, 256, 4), job(g.Q6_K, 100, 4)]) == 3   # the second job's K is not whole blocks
    assert run([job(g.Q4_K, 256, 4)], yt=g.Q8_0) == 2
    assert run([job(g.Q6_K, 256, 64)]) == 1                 # m = 64 is not decode-sized
    assert run([job(g.Q4_K, 256, 4, xq=0x20002)]) == 4      # q8_1 rows must be 4-byte aligned
    assert run([job(g.Q4_K, 256, 0)]) == 0                  # empty jobs are skipped
