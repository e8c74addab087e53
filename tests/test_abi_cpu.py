"""Host-side tests of the C ABI (no GPU needed): the library loads and exports
every symbol include/pa.h declares, pa_plan's partitioning, and the argument
checks that reject a call before anything is launched."""
import ctypes
import json
import os
import re
import subprocess

import pytest

import paged_kv_gqa_pa_gb300 as pa
from paged_kv_gqa_pa_gb300 import binding
from paged_kv_gqa_pa_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def built():
    pa_build.build()
    pa.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert {"pa_plan", "pa_decode", "pa_merge", "pa_get_error"} <= names
    lib = ctypes.CDLL(binding.library_path())
    for n in names:
        assert hasattr(lib, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()], check=True,
                        capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (pa_[a-z0-9_]+)$", nm, flags=re.M))
    assert names <= exported
    assert set(binding.EXPORTED) == names


def test_plan_struct_layout_matches_header():
    # Field names and order of the ctypes mirror equal the C struct's.
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    body = re.search(r"typedef struct pa_plan \{(.*?)\} pa_plan_t;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b(?:int|size_t|float)\s+([a-z_0-9]+)(?:\[\d+\])?\s*;", body)
    assert fields == [f for f, _ in binding.pa_plan_t._fields_]
    # 14 ints, a size_t, then 11 four-byte fields (kernel ... deep_ring).
    assert binding.pa_plan_t.workspace_bytes.offset == 56
    assert binding.pa_plan_t.kernel.offset == 64
    assert binding.pa_plan_t.parts_per_cta.offset == 68
    assert binding.pa_plan_t.prewait_prefetch.offset == 92
    assert binding.pa_plan_t.deep_ring.offset == 104
    assert ctypes.sizeof(binding.pa_plan_t) == 112


def test_status_strings_and_version():
    assert pa.pa_status_string(0) == "ok"
    assert "workspace" in pa.pa_status_string(4)
    assert pa.pa_version() >= 1


def test_plan_matches_the_pages_partition_counts():
    with open(os.path.join(HERE, "golden", "plan_partitions.json")) as f:
        spec = json.load(f)
    for c in spec["cases"]:
        L = c["context"]
        maxp = -(-L // 16)
        plan = pa.pa_plan(1, 8, 8, 128, 16, maxp, maxp, L, c["window"], c["partition_size"], 152)
        assert plan.num_partitions == c["num_partitions"]
        last = L - (plan.num_partitions - 1) * plan.partition_size
        assert last == c["last_partition_tokens"]


def test_plan_long_context_workload():
    plan = pa.pa_plan(4, 24, 4, 256, 16, 31250, 6250, 100000, 0, 512, 152)
    assert plan.num_partitions == 196 and plan.heads_per_cta == 6
    # 3136 one-partition CTAs would be ~10 waves of 304 resident CTAs; each
    # CTA serves 4 consecutive partitions instead (49 per group, 784 CTAs).
    assert plan.parts_per_cta == 4 and plan.ctas == 49 * 4 * 4
    # between 4 and 8 waves: 2 per CTA (B = 2: 1568 one-partition CTAs)
    half = pa.pa_plan(2, 24, 4, 256, 16, 31250, 6250, 100000, 0, 512, 152)
    assert half.parts_per_cta == 2 and half.ctas == 98 * 4 * 2
    # 4 per CTA would be 392 CTAs, 1.3 waves of 304: the slow case.
    # B = 1: 784 one-partition CTAs (2.6 waves); 4 per CTA makes one wave of
    # 196 CTAs that still covers all 152 SMs.
    one = pa.pa_plan(1, 24, 4, 256, 16, 6250, 6250, 100000, 0, 512, 152)
    assert one.parts_per_cta == 4 and one.ctas == 49 * 4
    # 50K tokens: 392 CTAs; 4 per CTA would leave SMs idle (100 CTAs), 2 per
    # CTA gives one wave of 196.
    mid = pa.pa_plan(1, 24, 4, 256, 16, 3125, 3125, 50000, 0, 512, 152)
    assert mid.parts_per_cta == 2 and mid.ctas == 49 * 4
    # The whole-wave split fills a wave to a little under its slots: 8 KV
    # heads at head_dim 128 (3 CTAs per SM, 456 slots) take 56 partitions,
    # not the 57 that would need every slot.
    l8 = pa.pa_plan(1, 32, 8, 128, 16, 8192, 8192, 131072, 0, 0, 152)
    assert l8.num_partitions == 56 and l8.ctas == 448
    # 32K tokens: 256 one-partition CTAs already fit in one wave.
    short = pa.pa_plan(1, 24, 4, 256, 16, 2048, 2048, 32768, 0, 512, 152)
    assert short.parts_per_cta == 1 and short.ctas == 64 * 4
    rows = 4 * 24 * 196
    assert plan.workspace_bytes >= 256 + rows * 4 * 2 + rows * 256 * 4


@pytest.mark.parametrize("num_sms", [1, 8, 152, 1000])
@pytest.mark.parametrize("B,Hkv,L,W", [(1, 1, 256, 0), (1, 8, 3060, 0), (8, 8, 4096, 0),
                                       (4, 4, 8192, 4096), (4, 4, 100000, 0), (1, 1, 17, 16)])
def test_auto_plan_is_consistent(num_sms, B, Hkv, L, W):
    maxp = -(-L // 16)
    plan = pa.pa_plan(B, Hkv * 4, Hkv, 128, 16, maxp * B, maxp, L, W, 0, num_sms)
    span = maxp if W == 0 else min(maxp, -(-(W - 1) // 16) + 1)
    if plan.balanced:
        # work-balanced: X CTAs per KV head over the batch; any lengths within
        # the bound fit X partitions of at most 2048 pages
        X = plan.balanced
        assert B >= 2 and plan.num_partitions == X and X > B
        assert B * span <= 2048 * (X - B)
        assert plan.partition_size // 16 == max(8, -(-(B * span) // (X - B)))
    else:
        assert plan.partition_size % 16 == 0 and plan.partition_size // 16 <= 256
        assert plan.num_partitions == -(-span // (plan.partition_size // 16))
    if plan.num_partitions == 1:
        assert plan.workspace_bytes == 256
    # The window bound covers every placement of the window.
    if W:
        worst = max(-(-Lb // 16) - (Lb - W) // 16 for Lb in range(W, L + 1))
        assert worst <= span


@pytest.mark.parametrize("args,status", [
    ((1, 8, 3, 128, 16, 10, 10, 100, 0, 0, 152), binding.PA_ERR_INVALID_ARG),   # Hq % Hkv
    ((1, 8, 8, 80, 16, 10, 10, 100, 0, 0, 152), binding.PA_ERR_UNSUPPORTED),    # head_dim
    ((1, 8, 8, 128, 32, 10, 10, 100, 0, 0, 152), binding.PA_ERR_UNSUPPORTED),   # page_size
    ((1, 8, 8, 128, 16, 10, 10, 100, 0, 24, 152), binding.PA_ERR_INVALID_ARG),  # S % 16
    ((1, 8, 8, 128, 16, 10, 10, 161, 0, 0, 152), binding.PA_ERR_INVALID_ARG),   # Lmax > table
    ((1, 18, 2, 128, 16, 10, 10, 100, 0, 0, 152), binding.PA_ERR_UNSUPPORTED),  # g = 9
    ((1, 8, 8, 128, 16, 10, 10, 100, 0, 32784, 152), binding.PA_ERR_UNSUPPORTED),  # S > 2048 pages
    ((1, 4, 1, 64, 16, 4200, 4200, 65552, 0, 16, 152), binding.PA_ERR_UNSUPPORTED),  # 4097 partitions
    ((-1, 8, 8, 128, 16, 10, 10, 100, 0, 0, 152), binding.PA_ERR_INVALID_ARG),
    ((1, 8, 8, 128, 16, 10, 10, 100, -1, 0, 152), binding.PA_ERR_INVALID_ARG),
])
def test_plan_rejects(args, status):
    with pytest.raises(pa.PAError) as e:
        pa.pa_plan(*args)
    assert e.value.status == status


def test_partition_size_limits_per_kernel():
    # A tensor-core CTA stages up to 2048 page ids, a CUDA-core CTA 256.
    ok = pa.pa_plan_ex(1, 8, 8, 128, 16, 4096, 4096, 65536, 0, 2048 * 16, 152)
    assert ok.partition_size == 2048 * 16 and ok.num_partitions == 2
    with pytest.raises(pa.PAError) as e:
        pa.pa_plan_ex(1, 8, 8, 128, 16, 4096, 4096, 65536, 0, 257 * 16, 152,
                      kernel=binding.PA_KERNEL_SIMT)
    assert e.value.status == binding.PA_ERR_UNSUPPORTED
    simt = pa.pa_plan_ex(1, 8, 8, 128, 16, 4096, 4096, 65536, 0, 256 * 16, 152,
                         kernel=binding.PA_KERNEL_SIMT)
    simt.partition_size = 512 * 16
    simt.num_partitions = 8
    assert _call_decode(simt) == binding.PA_ERR_INVALID_ARG


def _call_decode(plan, **over):
    fake = 0x10000  # aligned, never dereferenced: every case returns before a launch
    a = dict(q=fake, k=fake, v=fake, bt=fake, cl=fake, scale=0.1, window=plan.window, out=fake,
             lse=fake, ws=fake, stream=None)
    a.update(over)
    lib = pa.load()
    return lib.pa_decode(ctypes.byref(plan), a["q"], a["k"], a["v"], a["bt"], a["cl"],
                         ctypes.c_float(a["scale"]), a["window"], a["out"], a["lse"], a["ws"],
                         a["stream"])


def test_decode_argument_checks_return_before_launch():
    plan = pa.pa_plan(2, 8, 2, 128, 16, 100, 50, 800, 0, 64, 152)
    assert plan.num_partitions > 1
    assert _call_decode(plan, q=None) == binding.PA_ERR_INVALID_ARG
    assert _call_decode(plan, out=None) == binding.PA_ERR_INVALID_ARG
    assert _call_decode(plan, ws=None) == binding.PA_ERR_WORKSPACE
    assert _call_decode(plan, window=5) == binding.PA_ERR_INVALID_ARG
    assert _call_decode(plan, q=0x10002) == binding.PA_ERR_INVALID_ARG      # misaligned
    assert _call_decode(plan, ws=0x10008) == binding.PA_ERR_INVALID_ARG     # misaligned
    small = binding.pa_plan_t.from_buffer_copy(plan)
    small.workspace_bytes = 256
    assert _call_decode(small) == binding.PA_ERR_INVALID_ARG
    # the tensor-core kernel gives each of a CTA's partitions 4 / parts_per_cta warps
    for ppc in (3, 5, 8):
        odd = binding.pa_plan_t.from_buffer_copy(plan)
        odd.parts_per_cta = ppc
        assert _call_decode(odd) == binding.PA_ERR_INVALID_ARG, ppc
    bad = binding.pa_plan_t.from_buffer_copy(plan)
    bad.heads_per_cta = 3
    assert _call_decode(bad) == binding.PA_ERR_INVALID_ARG
    # The CUDA-core kernel has no head_dim-96 build, in any element type.
    p96 = pa.pa_plan(2, 8, 2, 96, 16, 100, 50, 800, 0, 64, 152)
    assert p96.kernel == binding.PA_KERNEL_MMA
    p96.kernel = binding.PA_KERNEL_SIMT
    assert _call_decode(p96) == binding.PA_ERR_UNSUPPORTED
    p96.dtype = binding.PA_DTYPE_BF16
    assert _call_decode(p96) == binding.PA_ERR_UNSUPPORTED
    # Rotary embedding: a negative base is invalid.
    rope_neg = binding.pa_plan_t.from_buffer_copy(plan)
    rope_neg.rope_theta = -1.0
    assert _call_decode(rope_neg) == binding.PA_ERR_INVALID_ARG
    f32_mma = binding.pa_plan_t.from_buffer_copy(plan)
    f32_mma.dtype = binding.PA_DTYPE_F32
    assert _call_decode(f32_mma) == binding.PA_ERR_UNSUPPORTED
    bad_dtype = binding.pa_plan_t.from_buffer_copy(plan)
    bad_dtype.dtype = 7
    assert _call_decode(bad_dtype) == binding.PA_ERR_INVALID_ARG
    empty = pa.pa_plan(0, 8, 2, 128, 16, 100, 50, 800, 0, 64, 152)
    assert _call_decode(empty) == binding.PA_OK   # nothing to do, nothing launched
    lib = pa.load()
    assert lib.pa_decode(None, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000, ctypes.c_float(1.0),
                         0, 0x10000, 0x10000, 0x10000, None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_merge(ctypes.byref(plan), 0x10000, 0x10000, 0x10000, None, None) == \
        binding.PA_ERR_WORKSPACE
    assert lib.pa_get_error(None, None, None) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_get_error_ex(None, None, 0, None) == binding.PA_ERR_INVALID_ARG


def test_binding_rejects_host_tensors():
    import torch
    plan = pa.pa_plan(1, 4, 1, 64, 16, 16, 16, 256, 0, 0, 152)
    t = torch.zeros(4, dtype=torch.float16)
    with pytest.raises(ValueError):
        pa.pa_decode(plan, t, t, t, t, t, 0.1, 0, t, t, t)


def test_plan_cta_count_saturates_instead_of_wrapping():
    # 65535 sequences x 64 KV heads x 1024 CTAs along the partitions is more
    # than an int holds; the informational count saturates
    p = pa.pa_plan(65535, 64, 64, 128, 16, 10**6, 4096, 65536, 0, 16, 152)
    assert p.ctas == 2**31 - 1 and p.num_partitions == 4096
    small = pa.pa_plan(2, 8, 2, 128, 16, 100, 50, 800, 0, 64, 152)
    assert small.ctas == small.batch * small.num_kv_heads * (
        -(-small.num_partitions // small.parts_per_cta))


def test_kernel_hash_ignores_comments_only():
    import bench
    code = "int f(int a) {\n  return a + 1;  // one\n}\n"
    assert bench.code_only(code) == bench.code_only(
        "/* header\n   lines */\nint f(int a) {\n\n  return a + 1;  // another note\n}\n")
    assert bench.code_only(code) != bench.code_only(code.replace("a + 1", "a + 2"))


def test_bench_kernel_source_lists_exist():
    import bench
    for kernel in bench.KERNEL_SOURCES:
        assert len(bench.kernel_src_sha(kernel)) == 16
    csrc = os.path.join(ROOT, "paged_kv_gqa_pa_gb300", "csrc")
    listed = {f for files in bench.KERNEL_SOURCES.values() for f in files}
    kernels = {f for f in os.listdir(csrc) if f.startswith("pa_attend")}
    assert kernels <= listed


def test_bench_counts_algorithmic_bytes_per_element_type():
    import bench
    from paged_kv_gqa_pa_gb300 import workloads
    for dtype, eb in (("f16", 2), ("bf16", 2), ("f32", 4)):
        c = workloads.make_case("b", 2, 4, 2, 64, [100, 40], seed=1, window=64, dtype=dtype)
        assert bench.kv_bytes(c) == 2 * eb * 2 * 64 * (64 + 40)


def test_plan_ex_picks_the_kernel_and_sizes_for_its_residency():
    args = (4, 32, 8, 128, 16, 10000, 2048, 32768, 0, 0, 152)
    f16 = pa.pa_plan_ex(*args)
    assert f16.kernel == binding.PA_KERNEL_MMA and f16.dtype == binding.PA_DTYPE_F16
    bf16 = pa.pa_plan_ex(*args, dtype=binding.PA_DTYPE_BF16)
    assert bf16.kernel == binding.PA_KERNEL_MMA and bf16.dtype == binding.PA_DTYPE_BF16
    f32 = pa.pa_plan_ex(*args, dtype=binding.PA_DTYPE_F32)
    assert f32.kernel == binding.PA_KERNEL_SIMT and f32.merge_in_kernel == 0
    rope = pa.pa_plan_ex(*args, rope_theta=10000.0)
    assert rope.kernel == binding.PA_KERNEL_MMA and rope.rope_theta == 10000.0
    # the rotary tensor-core instances run 2 CTAs per SM at D = 128 and 96
    # (the plain ones 3)
    assert rope.ctas < f16.ctas
    d96 = (4, 32, 8, 96, 16, 10000, 2048, 32768, 0, 0, 152)
    assert pa.pa_plan_ex(*d96, rope_theta=1e4).ctas < pa.pa_plan_ex(*d96).ctas
    # bf16 with a rotary embedding: the tensor-core kernel; fp32: the
    # CUDA-core kernel
    assert pa.pa_plan_ex(*args, rope_theta=1e4, dtype=binding.PA_DTYPE_BF16).kernel == \
        binding.PA_KERNEL_MMA
    assert pa.pa_plan_ex(*args, rope_theta=1e4, dtype=binding.PA_DTYPE_F32).kernel == \
        binding.PA_KERNEL_SIMT
    wide_args = (4, 24, 4, 256, 16, 10000, 2048, 32768, 0, 0, 152)
    # head dim 256: the tensor-core rotary instances too (3 ring stages, 2 CTAs per SM)
    assert pa.pa_plan_ex(*wide_args, rope_theta=1e4).kernel == binding.PA_KERNEL_MMA
    assert pa.pa_plan_ex(*wide_args, rope_theta=1e4, dtype=binding.PA_DTYPE_BF16).kernel == \
        binding.PA_KERNEL_MMA
    assert pa.pa_plan_ex(*wide_args, rope_theta=1e4, dtype=binding.PA_DTYPE_F32).kernel == \
        binding.PA_KERNEL_SIMT
    # fp32 at D = 256 keeps one CTA per SM, so its automatic grid is smaller
    wide = (4, 24, 4, 256, 16, 10000, 2048, 32768, 0, 0, 152)
    assert (pa.pa_plan_ex(*wide, dtype=binding.PA_DTYPE_F32).ctas <
            pa.pa_plan_ex(*wide).ctas)
    for kw, st in ((dict(dtype=binding.PA_DTYPE_F32, kernel=binding.PA_KERNEL_MMA),
                    binding.PA_ERR_UNSUPPORTED),
                   (dict(rope_theta=1e4, kernel=binding.PA_KERNEL_MMA,
                         dtype=binding.PA_DTYPE_F32), binding.PA_ERR_UNSUPPORTED),
                   (dict(dtype=9), binding.PA_ERR_INVALID_ARG),
                   (dict(kernel=7), binding.PA_ERR_INVALID_ARG),
                   (dict(rope_theta=-2.0), binding.PA_ERR_INVALID_ARG)):
        with pytest.raises(pa.PAError) as e:
            pa.pa_plan_ex(*args, **kw)
        assert e.value.status == st
    # bf16 on the CUDA-core kernel, with or without a rotary embedding
    for kw in (dict(dtype=binding.PA_DTYPE_BF16, kernel=binding.PA_KERNEL_SIMT),
               dict(dtype=binding.PA_DTYPE_BF16, kernel=binding.PA_KERNEL_SIMT, rope_theta=1e4)):
        assert pa.pa_plan_ex(*args, **kw).kernel == binding.PA_KERNEL_SIMT
    d96 = (4, 32, 8, 96, 16, 10000, 2048, 32768, 0, 0, 152)
    with pytest.raises(pa.PAError) as e:
        pa.pa_plan_ex(*d96, dtype=binding.PA_DTYPE_BF16, kernel=binding.PA_KERNEL_SIMT)
    assert e.value.status == binding.PA_ERR_UNSUPPORTED
    with pytest.raises(pa.PAError):
        pa.pa_plan_ex(4, 32, 8, 96, 16, 10000, 2048, 32768, 0, 0, 152,
                      kernel=binding.PA_KERNEL_SIMT)


def test_plan_picks_the_cluster_merge_for_one_wave_splits():
    # Gemma-2-2b shape: 16 groups, 257 window pages; one wave of 2-per-SM
    # tensor-core CTAs holds 19 clusters of 13 CTAs but only 14 of 14..16, so
    # each group is a 13-CTA cluster of 20-page partitions.
    gemma = pa.pa_plan_ex(4, 8, 4, 256, 16, 3000, 512, 8192, 4096, 0, 152)
    assert gemma.cluster == gemma.num_partitions == 13
    assert gemma.parts_per_cta == 1 and gemma.merge_in_kernel == 0
    assert gemma.partition_size == 20 * 16 and gemma.ctas == 16 * 13
    assert gemma.prewait_prefetch == 2
    # Llama-3.2-1B shape: 8 groups, 192 pages, 16 partitions of 12 pages.
    llama = pa.pa_plan_ex(1, 32, 8, 64, 16, 300, 192, 3060, 0, 0, 152)
    assert llama.cluster == 16 and llama.partition_size == 12 * 16
    # 100 000 tokens do not fit 16 partitions: many partitions and the merge kernel.
    long = pa.pa_plan_ex(4, 24, 4, 256, 16, 30000, 6250, 100000, 0, 0, 152)
    assert long.cluster == 0 and long.num_partitions > 16
    # The CUDA-core kernel never clusters; an explicit partition size never does.
    assert pa.pa_plan_ex(4, 8, 4, 256, 16, 3000, 512, 8192, 4096, 0, 152,
                         kernel=binding.PA_KERNEL_SIMT).cluster == 0
    assert pa.pa_plan_ex(4, 8, 4, 256, 16, 3000, 512, 8192, 4096, 512, 152).cluster == 0
    # A short context stays unsplit.
    assert pa.pa_plan_ex(1, 4, 1, 64, 16, 64, 16, 256, 0, 0, 152).cluster == 0
    # An explicit SM count other than the measured part's scales the table's
    # fill fraction: on 76 SMs a wave holds 17 clusters of 8 (>= 16 groups)
    # but only 15 of 9.
    half = pa.pa_plan_ex(4, 8, 4, 256, 16, 3000, 512, 8192, 4096, 0, 76)
    assert half.cluster == half.num_partitions == 8


def test_cluster_plan_checks_return_before_launch():
    plan = pa.pa_plan_ex(4, 8, 4, 256, 16, 3000, 512, 8192, 4096, 0, 152)
    assert plan.cluster == 13
    for field, value in (("cluster", 17), ("cluster", 8), ("cluster", -1),
                         ("parts_per_cta", 2), ("merge_in_kernel", 1),
                         ("kernel", binding.PA_KERNEL_SIMT)):
        bad = binding.pa_plan_t.from_buffer_copy(plan)
        setattr(bad, field, value)
        assert _call_decode(bad) == binding.PA_ERR_INVALID_ARG, (field, value)
    # pa_merge has nothing to do after a clustered partition kernel.
    lib = pa.load()
    assert lib.pa_merge(ctypes.byref(plan), 0x10000, 0x10000, 0x10000, 0x10000, None) == \
        binding.PA_OK


def test_partition_count_limit():
    # the merge kernel reduces at most 4096 partitions per head
    ok = pa.pa_plan(1, 4, 1, 64, 16, 4200, 4096, 65536, 0, 16, 152)
    assert ok.num_partitions == 4096


STATIC_BYTES = 32 << 20  # PA_STATIC_WORKSPACE_BYTES in include/pa.h


def test_static_entry_point_checks_the_plan_before_touching_the_gpu():
    """pa_decode_static runs pa_decode's plan checks, then sizes the workspace
    extent from the plan's shapes, all on the host: these calls are rejected
    on a machine without a GPU, so none of them reaches a CUDA call."""
    lib = pa.load()
    fake = ctypes.c_void_p(0x10000)  # never dereferenced

    def call(plan):
        return lib.pa_decode_static(ctypes.byref(plan), fake, fake, fake, fake, fake,
                                    ctypes.c_float(0.1), plan.window, fake, fake, None)

    plan = pa.pa_plan(4, 32, 8, 128, 16, 4000, 256, 4096, 0, 256, 152)
    assert plan.num_partitions > 1 and plan.workspace_bytes <= STATIC_BYTES
    # A control region claimed larger than the whole scratch (a stale or
    # hand-edited plan) never reaches the clearing memset.
    huge = binding.pa_plan_t.from_buffer_copy(plan)
    huge.ctrl_bytes = 64 << 20
    assert call(huge) == binding.PA_ERR_INVALID_ARG
    huge.workspace_bytes = 80 << 20
    assert call(huge) == binding.PA_ERR_WORKSPACE
    # A control region too small for the arrival counters the launch uses
    # (heads_per_cta edited after pa_plan: 4 head chunks per KV head instead of 1).
    chunks = binding.pa_plan_t.from_buffer_copy(plan)
    chunks.heads_per_cta = 1
    chunks.merge_in_kernel = 0
    assert call(chunks) == binding.PA_ERR_INVALID_ARG
    negative = binding.pa_plan_t.from_buffer_copy(plan)
    negative.ctrl_bytes = -1
    assert call(negative) == binding.PA_ERR_INVALID_ARG
    # A plan whose partials need more than the built-in scratch.
    big = pa.pa_plan(4, 64, 8, 256, 16, 1 << 16, 4096, 65536, 0, 16, 152)
    assert big.workspace_bytes > STATIC_BYTES
    assert call(big) == binding.PA_ERR_WORKSPACE
    # Everything else pa_decode rejects, pa_decode_static rejects the same way.
    bad = binding.pa_plan_t.from_buffer_copy(plan)
    bad.parts_per_cta = 3
    assert call(bad) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_decode_static(None, fake, fake, fake, fake, fake, ctypes.c_float(0.1), 0,
                                fake, fake, None) == binding.PA_ERR_INVALID_ARG


def test_plan_rejects_control_bytes_that_miss_counters():
    plan = pa.pa_plan(4, 32, 8, 128, 16, 4000, 256, 4096, 0, 256, 152)
    edited = binding.pa_plan_t.from_buffer_copy(plan)
    edited.heads_per_cta = 1
    edited.merge_in_kernel = 0
    # 4 x 32 groups of counters need more control bytes than the 4 x 8 of the plan
    assert _call_decode(edited) == binding.PA_ERR_INVALID_ARG
    # a control region larger than the workspace is inconsistent too
    over = binding.pa_plan_t.from_buffer_copy(plan)
    over.ctrl_bytes = int(over.workspace_bytes) + 256
    assert _call_decode(over) == binding.PA_ERR_INVALID_ARG


def test_balanced_plans():
    """partition_size = PA_PARTITION_BALANCED: X CTAs per (KV head, head
    chunk) over the whole batch, one wave, the last-CTA merge."""
    BAL = binding.PA_PARTITION_BALANCED
    # the ragged batch-8 shape: 8 groups, 3 CTAs per SM -> 448 of 456 slots
    p = pa.pa_plan_ex(8, 32, 8, 128, 16, 1250, 256, 4096, 0, BAL, 152)
    assert p.balanced == 56 and p.num_partitions == 56 and p.ctas == 56 * 8
    assert p.merge_in_kernel == 1 and p.cluster == 0 and p.parts_per_cta == 1
    # the largest partition any lengths within the bound can give: 8 x 256 pages over 48
    assert p.partition_size == 16 * 43
    assert p.workspace_bytes >= 8 * 32 * 56 * (128 + 2) * 4
    # none for the CUDA-core kernel, a rotary embedding, more than 128 sequences,
    # or a bound whose pages could not fit X partitions of 2048 pages
    for args, kw in (((8, 32, 8, 128, 16, 1250, 256, 4096, 0, BAL, 152),
                      dict(kernel=binding.PA_KERNEL_SIMT)),
                     ((8, 32, 8, 128, 16, 1250, 256, 4096, 0, BAL, 152),
                      dict(rope_theta=10000.0)),
                     ((129, 8, 2, 64, 16, 9000, 64, 1024, 0, BAL, 152), {}),
                     ((8, 32, 8, 128, 16, 200000, 16384, 262144, 0, BAL, 152), {})):
        with pytest.raises(pa.PAError) as e:
            pa.pa_plan_ex(*args, **kw)
        assert e.value.status == binding.PA_ERR_UNSUPPORTED, (args, kw)
    # edits that break the plan's rules are rejected before any launch
    for field, value in (("cluster", 8), ("parts_per_cta", 2),
                         ("balanced", 8), ("balanced", -1), ("rope_theta", 10000.0),
                         ("kernel", binding.PA_KERNEL_SIMT)):
        bad = binding.pa_plan_t.from_buffer_copy(p)
        setattr(bad, field, value)
        assert _call_decode(bad) == binding.PA_ERR_INVALID_ARG, (field, value)
    # a fixed-size plan never sets it
    assert pa.pa_plan_ex(8, 32, 8, 128, 16, 1250, 256, 4096, 0, 512, 152).balanced == 0
    # The merge: the last CTA of each group, unless one group could leave it
    # more than 128 KiB of partials (X - B + 1 partials of G x D floats).
    wide = pa.pa_plan_ex(4, 64, 8, 128, 16, 5000, 3125, 50000, 0, BAL, 152)
    assert wide.balanced == 56 and (56 - 4 + 1) * 8 * 128 * 4 > 128 << 10
    assert wide.merge_in_kernel == 0
    narrow = pa.pa_plan_ex(16, 32, 8, 128, 16, 5000, 750, 12000, 0, BAL, 152)
    assert narrow.balanced == 56 and (56 - 16 + 1) * 4 * 128 * 4 <= 128 << 10
    assert narrow.merge_in_kernel == 1


def test_rotary_plans_merge_in_the_last_cta_when_partials_are_small():
    """Rotary instances with fixed partitions: the last CTA of each group
    merges when a group's partials (P x G x D floats) are at most 128 KiB,
    the merge kernel otherwise."""
    def plan(B, Hq, Hkv, D, L):
        pages = -(-L // 16)
        return pa.pa_plan_ex(B, Hq, Hkv, D, 16, B * pages + 8, pages, L, 0, 0, 152,
                             rope_theta=1e4)
    small = plan(4, 24, 4, 256, 32768)  # P 18: 18 x 6 x 256 x 4 B = 110.6 KB
    assert small.cluster == 0 and small.num_partitions * 6 * 256 * 4 <= 128 << 10
    assert small.merge_in_kernel == 1
    big = plan(1, 24, 4, 256, 65536)    # P 75: 460.8 KB
    assert big.cluster == 0 and big.num_partitions * 6 * 256 * 4 > 128 << 10
    assert big.merge_in_kernel == 0
    # without rotary embedding the same small shape keeps the merge kernel
    plain = pa.pa_plan_ex(4, 24, 4, 256, 16, 4 * 2048 + 8, 2048, 32768, 0, 1824, 152)
    assert plain.num_partitions == 18 and plain.merge_in_kernel == 0


def test_deep_ring_cluster_instance_for_small_cluster_grids():
    """Cluster plans of plain head dims 96 and 128 whose grid has at most one
    CTA per SM take the instance with deeper page rings (2 CTAs per SM); at
    head dim 256 (1 CTA per SM) grids of at most half the SMs."""
    def plan(B, D, L, **kw):
        pages = -(-L // 16)
        return pa.pa_plan_ex(B, 32, 8, D, 16, B * pages + 8, pages, L, 0, 0, 152, **kw)
    for D in (96, 128):
        one = plan(1, D, 16384)
        assert one.cluster == 16 and one.ctas == 128 and one.deep_ring == 1
    # a grid that needs more than one CTA per SM, other head dims, rotary
    # plans and plans without a cluster keep the default instance
    assert plan(8, 128, 4096).cluster == 6 and plan(8, 128, 4096).deep_ring == 0
    assert plan(2, 128, 8192).ctas > 152 and plan(2, 128, 8192).deep_ring == 0
    assert plan(1, 64, 16384).cluster == 16 and plan(1, 64, 16384).deep_ring == 0
    # head dim 256: 1 CTA per SM, only for grids of at most half the SMs
    def plan256(B, Hq, Hkv, L, window=0):
        pages = -(-L // 16)
        return pa.pa_plan_ex(B, Hq, Hkv, 256, 16, B * pages + 8, pages, L, window, 0, 152)
    assert plan256(1, 24, 4, 16384).ctas == 64 and plan256(1, 24, 4, 16384).deep_ring == 1
    assert plan256(1, 16, 8, 8192).ctas == 128 and plan256(1, 16, 8, 8192).deep_ring == 0
    assert plan256(4, 8, 4, 8192, 4096).deep_ring == 0  # the Gemma-2 workload
    assert plan(1, 128, 16384, rope_theta=1e4).deep_ring == 0
    assert plan(1, 128, 32768).cluster == 0 and plan(1, 128, 32768).deep_ring == 0
    # the ABI: 0 or 1; with a cluster, 1 only where the instance exists; it is
    # ignored without a cluster
    ok = plan(1, 128, 16384)
    for field, value, status in (("deep_ring", 2, binding.PA_ERR_INVALID_ARG),
                                 ("deep_ring", -1, binding.PA_ERR_INVALID_ARG)):
        bad = binding.pa_plan_t.from_buffer_copy(ok)
        setattr(bad, field, value)
        assert _call_decode(bad) == status
    rope = plan(1, 128, 16384, rope_theta=1e4)
    assert rope.cluster > 1
    rope.deep_ring = 1
    assert _call_decode(rope) == binding.PA_ERR_INVALID_ARG
    d64 = plan(1, 64, 16384)
    d64.deep_ring = 1
    assert _call_decode(d64) == binding.PA_ERR_INVALID_ARG
