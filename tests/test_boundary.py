"""The C ABI boundary without a GPU: the library loads, exports every symbol the
header declares, plans workspaces on the host, and rejects bad calls before
any CUDA work (status codes and messages)."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_decode_15_gb300 as pkd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkd.h")


@pytest.fixture(scope="module")
def lib():
    pkd.build()
    return pkd.load_library()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert set(declared_symbols()) == set(pkd.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version(lib):
    assert pkd.version() == 10000


def test_workspace_plan_is_a_host_function(lib):
    # gqa decode, B=64, Hq=32, Hkv=8, D=128, P=16, capacity 4096
    n = pkd.workspace_size(64, 1, 32, 8, 128, 16, 4096, pkd.BF16)
    assert n > 0 and n % 256 == 0
    # more splits for longer capacity
    assert pkd.workspace_size(8, 1, 64, 8, 128, 64, 131072, pkd.FP8_E4M3) > 0
    # chunked grid, explicit chunk: 4096 / 256 = 16 splits -> partials [512 units, 16, 4 rows, 128] fp32
    m = pkd.workspace_size(64, 1, 32, 8, 128, 16, 4096, pkd.BF16, chunk_tokens=256, flags=pkd.FLAG_GRID)
    assert m >= 512 * 16 * 4 * 128 * 4
    # flat partition: two partial slots per worker warp, independent of the lengths
    f1 = pkd.workspace_size(8, 1, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_FLAT)
    f2 = pkd.workspace_size(8, 1, 32, 8, 128, 16, 131072, pkd.BF16, flags=pkd.FLAG_FLAT)
    assert f1 == f2 and f1 >= 2048 * 2 * 4 * 128 * 4
    # 16-bit caches with M <= 16 take the chunked grid by default ...
    assert n == pkd.workspace_size(64, 1, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_GRID)
    # ... fp8 caches too ...
    assert pkd.workspace_size(64, 1, 32, 8, 128, 16, 4096, pkd.FP8_E4M3) == \
        pkd.workspace_size(64, 1, 32, 8, 128, 16, 4096, pkd.FP8_E4M3, flags=pkd.FLAG_GRID)
    # ... 16-bit M > 16 (dense or causal) takes the tcgen05 kernel: chunks
    # of at most 2048 keys, and a unit of n chunks in at most n + 1 pieces
    # (CTA shares at least a chunk long), a partial slot of 32 rows each ...
    w = pkd.workspace_size(64, 8, 32, 8, 128, 16, 8192, pkd.BF16)
    assert 512 * 5 * 32 * 128 * 4 <= w < 512 * 6 * 32 * 128 * 4
    assert w == pkd.workspace_size(64, 8, 32, 8, 128, 16, 8192, pkd.BF16, chunk_tokens=2048)
    assert w < pkd.workspace_size(64, 8, 32, 8, 128, 16, 8192, pkd.BF16, chunk_tokens=1024)
    assert w == pkd.workspace_size(64, 8, 32, 8, 128, 16, 8192, pkd.BF16, flags=pkd.FLAG_CAUSAL)
    # ... forced grids keep the warp-pair kernel (as few chunks as the 4096-key
    # limit allows: 8192 keys -> 2 chunks -> partials [512, 2, 32, 128])
    g = pkd.workspace_size(64, 8, 32, 8, 128, 16, 8192, pkd.BF16, flags=pkd.FLAG_CAUSAL | pkd.FLAG_GRID)
    assert g == pkd.workspace_size(64, 8, 32, 8, 128, 16, 8192, pkd.BF16, chunk_tokens=4096, flags=pkd.FLAG_GRID)
    assert 512 * 2 * 32 * 128 * 4 <= g < 512 * 3 * 32 * 128 * 4
    # ... while fp8 with M > 16 stays on the flat partition whatever the lengths
    assert pkd.workspace_size(64, 8, 32, 8, 128, 16, 4096, pkd.FP8_E4M3) == \
        pkd.workspace_size(64, 8, 32, 8, 128, 16, 131072, pkd.FP8_E4M3)
    # the e4m3 grid takes the same rule: 64 units of 131072 keys -> 32 chunks of 4096
    assert pkd.workspace_size(8, 1, 64, 8, 128, 64, 131072, pkd.FP8_E4M3) == \
        pkd.workspace_size(8, 1, 64, 8, 128, 64, 131072, pkd.FP8_E4M3, chunk_tokens=4096)
    assert pkd.workspace_size(8, 1, 64, 8, 128, 64, 131072, pkd.FP8_E4M3) != \
        pkd.workspace_size(8, 1, 64, 8, 128, 64, 131072, pkd.FP8_E4M3, chunk_tokens=4032)
    # batches above the flat kernel's table size use the chunked grid
    assert pkd.workspace_size(2048, 1, 32, 8, 128, 16, 4096, pkd.BF16) == \
        pkd.workspace_size(2048, 1, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_GRID)


@pytest.mark.parametrize("args,needle", [
    ((2, 1, 6, 4, 128, 16, 100, pkd.BF16), "multiple of num_kv_heads"),
    ((2, 1, 8, 2, 96, 16, 100, pkd.BF16), "head_dim"),
    ((2, 1, 8, 2, 128, 8, 100, pkd.BF16), "page_size"),
    ((2, 4, 32, 8, 128, 16, 100, pkd.FP8_E4M3, 0, 0, pkd.FLAG_FMA), "fp8"),
    ((2, 8, 32, 8, 128, 16, 100, pkd.FP8_E4M3, 0, 0, pkd.FLAG_GRID), "fp8"),
    ((2, 16, 32, 8, 128, 16, 100, pkd.BF16), "> 32"),
    ((2, 1, 8, 2, 64, 16, 100, pkd.FP8_E4M3), "head_dim 128"),
])
def test_unsupported_plans_are_rejected_with_a_reason(lib, args, needle):
    with pytest.raises(pkd.PkdError) as e:
        pkd.workspace_size(*args)
    assert needle in str(e.value)


def test_chunk_must_be_a_page_multiple(lib):
    with pytest.raises(pkd.PkdError):
        pkd.workspace_size(2, 1, 8, 2, 128, 16, 100, pkd.BF16, chunk_tokens=24)


def _decode_call(lib, **over):
    a = dict(q=None, q_dt=pkd.BF16, kv=None, kv_dt=pkd.BF16, num_pages=8, bt=None, bt_stride=4, lens=None, B=2,
             sq=1, Hq=4, Hkv=2, D=64, P=16, max_kv_len=64, scale=0.125, qs=1.0, ks=1.0, vs=1.0, window=0,
             out=None, out_dt=pkd.BF16, lse=None, ws=None, ws_bytes=1 << 20, chunk=0, flags=0, stream=None)
    a.update(over)
    return lib.pkd_paged_decode(*a.values())


def test_zero_batch_is_ok_without_a_gpu(lib):
    assert _decode_call(lib, B=0) == pkd.OK


def test_null_pointers_are_einval(lib):
    assert _decode_call(lib) == pkd.EINVAL
    assert b"null" in lib.pkd_last_error()


def test_host_io_refuses_memory_not_registered_with_cuda(lib):
    # plain host buffers: refused by the pointer check, before any CUDA work
    bufs = [ctypes.create_string_buffer(1 << 16) for _ in range(6)]
    a = [ctypes.c_void_p((ctypes.addressof(b) + 255) // 256 * 256) for b in bufs]
    st = _decode_call(lib, q=a[0], kv=a[1], bt=a[2], lens=a[3], out=a[4], ws=a[5], flags=pkd.FLAG_HOST_IO)
    assert st == pkd.EINVAL
    assert b"PKD_FLAG_HOST_IO: q is not pinned host memory" in lib.pkd_last_error()


def test_host_io_plans_run_the_chunked_grid_for_tcgen05_shapes(lib):
    shape = (50, 8, 32, 8, 128, 16, 2048, pkd.BF16)
    assert pkd.FLAG_HOST_IO == 128
    assert pkd.kernel_name(*shape) == "persistent tcgen05 kernel, TMEM accumulators"
    assert pkd.kernel_name(*shape, flags=pkd.FLAG_HOST_IO) == pkd.kernel_name(*shape, flags=pkd.FLAG_GRID)
    assert pkd.workspace_size(*shape, flags=pkd.FLAG_HOST_IO) == pkd.workspace_size(*shape, flags=pkd.FLAG_GRID)
    assert pkd.kernel_name(64, 1, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_HOST_IO) == \
        pkd.kernel_name(64, 1, 32, 8, 128, 16, 4096, pkd.BF16)


def test_mismatched_q_and_cache_types(lib):
    assert _decode_call(lib, q_dt=pkd.FP16) == pkd.EUNSUPPORTED


def test_bad_out_dtype(lib):
    assert _decode_call(lib, out_dt=pkd.FP8_E4M3) == pkd.EUNSUPPORTED


def test_misaligned_and_small_workspace(lib):
    fake = 1 << 20
    kw = dict(q=fake, kv=fake, bt=fake, lens=fake, out=fake, ws=fake)
    assert _decode_call(lib, **dict(kw, kv=fake + 8)) == pkd.EINVAL
    assert b"misaligned" in lib.pkd_last_error()
    assert _decode_call(lib, **dict(kw, ws_bytes=256)) == pkd.EINVAL
    assert b"workspace too small" in lib.pkd_last_error()
    assert _decode_call(lib, **dict(kw, bt_stride=2)) == pkd.EINVAL
    assert b"block_table_stride" in lib.pkd_last_error()


def test_segmented_validation(lib):
    seg = lib.pkd_segmented_attention
    P = None
    # fp8 is not a segmented dtype
    assert seg(P, P, P, pkd.FP8_E4M3, P, P, 4, 8, 2, 128, 2, 16, 16, P, P, P, P) == pkd.EUNSUPPORTED
    # bs not a multiple of 8
    assert seg(P, P, P, pkd.BF16, P, P, 4, 8, 2, 128, 2, 12, 16, P, P, P, P) == pkd.EUNSUPPORTED
    # n == 0 is a no-op
    assert seg(P, P, P, pkd.BF16, P, P, 0, 8, 2, 128, 2, 16, 16, P, P, P, P) == pkd.OK
    # null inputs
    assert seg(P, P, P, pkd.BF16, P, P, 4, 8, 2, 128, 2, 16, 16, P, P, P, P) == pkd.EINVAL


def test_lse_merge_validation(lib):
    m = lib.pkd_lse_merge
    assert m(None, None, None, None, 0, 4, 2, 64, None, pkd.FP32, None, None) == pkd.OK
    assert m(None, None, None, None, 3, 4, 2, 64, None, pkd.FP32, None, None) == pkd.EINVAL
    assert m(None, None, None, None, 3, 4, 2, 512, None, pkd.FP32, None, None) == pkd.EUNSUPPORTED


def test_kernel_name_follows_the_plan(lib):
    args = (64, 1, 32, 8, 128, 16, 4096)
    assert pkd.kernel_name(*args, pkd.BF16) == "chunked grid, tensor cores"
    assert pkd.kernel_name(*args, pkd.BF16, flags=pkd.FLAG_FLAT) == "persistent flat partition, tensor cores"
    assert pkd.kernel_name(8, 1, 32, 8, 128, 16, 4096, pkd.BF16) == "chunked grid, tensor cores"
    assert pkd.kernel_name(8, 8, 32, 8, 128, 16, 4096, pkd.BF16) == "persistent tcgen05 kernel, TMEM accumulators"
    assert pkd.kernel_name(8, 8, 32, 8, 128, 16, 4096, pkd.FP16) == "persistent tcgen05 kernel, TMEM accumulators"
    assert pkd.kernel_name(8, 8, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_CAUSAL) == \
        "persistent tcgen05 kernel, TMEM accumulators"
    assert pkd.kernel_name(8, 8, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_CAUSAL | pkd.FLAG_GRID) == \
        "chunked grid, tensor cores"
    assert pkd.kernel_name(8, 8, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_GRID) == "chunked grid, tensor cores"
    assert pkd.kernel_name(8, 8, 32, 8, 64, 16, 4096, pkd.BF16) == "chunked grid, tensor cores"
    assert pkd.kernel_name(8, 8, 32, 8, 128, 16, 8192, pkd.BF16, chunk_tokens=4096) == "chunked grid, tensor cores"
    assert pkd.kernel_name(2048, 8, 32, 8, 128, 16, 4096, pkd.BF16) == "chunked grid, tensor cores"
    assert pkd.kernel_name(513, 8, 32, 8, 128, 16, 4096, pkd.BF16) == "chunked grid, tensor cores"
    assert pkd.kernel_name(8, 8, 32, 8, 128, 16, 4096, pkd.FP8_E4M3) == "persistent flat partition, tensor cores"
    assert pkd.kernel_name(*args, pkd.BF16, flags=pkd.FLAG_FMA | pkd.FLAG_GRID) == "chunked grid, CUDA cores"
    assert pkd.kernel_name(*args, pkd.FP8_E4M3) == "chunked grid, tensor cores"
    assert pkd.kernel_name(64, 8, 32, 8, 128, 16, 4096, pkd.FP8_E4M3) == "persistent flat partition, tensor cores"
    assert pkd.kernel_name(*args, pkd.FP8_E4M3, flags=pkd.FLAG_GRID) == "chunked grid, tensor cores"
    assert pkd.kernel_name(*args, pkd.FP8_E4M3, flags=pkd.FLAG_GRID | pkd.FLAG_FMA) == "chunked grid, CUDA cores"
    assert pkd.kernel_name(2048, 1, 32, 8, 128, 16, 4096, pkd.FP8_E4M3) == "chunked grid, tensor cores"
    with pytest.raises(pkd.PkdError, match="head_dim"):
        pkd.kernel_name(2, 1, 8, 2, 96, 16, 100, pkd.BF16)
    with pytest.raises(pkd.PkdError, match="exclude"):
        pkd.kernel_name(*args, pkd.BF16, flags=pkd.FLAG_FLAT | pkd.FLAG_GRID)
    assert pkd.kernel_name(*args, pkd.BF16, flags=pkd.FLAG_BALANCED) == "persistent per-CTA partition, tensor cores"
    with pytest.raises(pkd.PkdError, match="16-bit"):
        pkd.kernel_name(*args, pkd.FP8_E4M3, flags=pkd.FLAG_BALANCED)
    # the per-CTA partition: two partial slots per CTA (<= 512 CTAs), whatever the lengths or the batch
    b1 = pkd.workspace_size(64, 1, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_BALANCED)
    b2 = pkd.workspace_size(64, 1, 32, 8, 128, 16, 131072, pkd.BF16, flags=pkd.FLAG_BALANCED)
    assert b1 == b2 and b1 >= 512 * 2 * 4 * 128 * 4
    assert pkd.kernel_name(4096, 8, 32, 8, 128, 16, 4096, pkd.BF16, flags=pkd.FLAG_BALANCED).startswith("persistent")


def test_launch_setup_is_kept_per_device(tmp_path):
    """The per-device memo of kernel launch set-up, driven from eight host
    threads on two stub devices (compiled with g++, no GPU)."""
    src = os.path.join(ROOT, "tests", "device_state_check.cpp")
    exe = str(tmp_path / "device_state_check")
    csrc = os.path.join(ROOT, "paged_kv_decode_15_gb300", "csrc")
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-pthread", "-I", csrc, src, "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr


def test_page_division_by_magic_number_is_exact(tmp_path):
    """tok / P and tok % P as the kernels compute them (multiply and shift)
    against the integer division, for every page size up to 4096."""
    src = os.path.join(ROOT, "tests", "page_math_check.cpp")
    exe = str(tmp_path / "page_math_check")
    csrc = os.path.join(ROOT, "paged_kv_decode_15_gb300", "csrc")
    r = subprocess.run(["g++", "-std=c++17", "-O2", "-I", csrc, src, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
