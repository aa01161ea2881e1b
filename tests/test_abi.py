"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports
every function include/ds_topk.h declares, and rejects bad arguments before it touches
the device."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds_topk.h")


@pytest.fixture(scope="module")
def lib():
    from top_selection_gb300 import build
    build.build()
    import top_selection_gb300 as ds
    return ds.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(ds_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["ds_topk", "ds_topk_ex", "ds_get_plan", "ds_workspace_bytes",
                 "ds_get_device_status", "ds_status_string", "ds_version", "ds_block_order",
                 "ds_wait_probe"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\b[TW]\s+(ds_\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_header_compiles_as_c():
    src = '#include "ds_topk.h"\nint main(void){ ds_status s = DS_OK; (void)s; return 0; }\n'
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I" + os.path.join(ROOT, "include"),
                    "-x", "c", "-"], input=src, text=True, check=True)


def test_version_and_status_strings(lib):
    import top_selection_gb300 as ds
    assert "sm_103a" in ds.ds_version()
    for code in range(8):
        assert ds.ds_status_string(code)


# Pointers below are never dereferenced: argument checks run before any CUDA call.
P = 1 << 20   # a 16-byte aligned fake device address


@pytest.mark.parametrize("args,want", [
    (dict(dtype=2), 1),                         # unknown dtype
    (dict(k=0), 1),
    (dict(k=1001), 1),                          # k > N
    (dict(B=-1), 1),                            # (0 asks for the library's choice)
    (dict(B2=-1), 1),
    (dict(N=0), 1),
    (dict(rows=-1), 1),
    (dict(row_stride=999), 1),                  # stride < N
    (dict(x=0), 1),                             # null input
    (dict(out_idx=0), 1),
    (dict(x=P + 8), 2),                         # misaligned input
    (dict(out_vals=P + 4), 2),
    (dict(row_stride=1004), 2),                 # 1004 * 2 bytes is not a multiple of 16
    (dict(N=5000, row_stride=5000, k=4097), 3), # k above 4096
    (dict(B=1001), 3),                          # B * 2 bytes not a multiple of 16
    (dict(rows=0), 0),                          # nothing to do
])
def test_host_validation(lib, args, want):
    import top_selection_gb300 as ds
    a = dict(x=P, dtype=0, rows=2, N=1000, row_stride=1024, k=8, B=64, B2=64, seed=1,
             out_vals=P, out_idx=P)
    a.update(args)
    st = ds.ds_topk(a["x"], a["dtype"], a["rows"], a["N"], a["row_stride"], a["k"], a["B"], a["B2"],
                    a["seed"], a["out_vals"], a["out_idx"], 0)
    assert st == want


def test_fp32_alignment_rules(lib):
    import top_selection_gb300 as ds
    # fp32: B*4 must be a multiple of 16 -> B % 4 == 0; stride*4 % 16 -> stride % 4 == 0
    assert ds.ds_topk(P, 1, 2, 100, 102, 4, 8, 8, 0, P, P, 0) == 2
    assert ds.ds_topk(P, 1, 1, 100, 100, 4, 10, 8, 0, P, P, 0) == 3
    assert ds.ds_topk(P, 1, 0, 100, 100, 4, 8, 8, 0, P, P, 0) == 0


_PLAN_SCRIPT = r"""
import json, top_selection_gb300 as ds
ds.load()
shapes = {"indexer": (0, 64, 131072, 512, 4096, 4096), "sampler": (1, 256, 129280, 512, 8192, 4096),
          "sampler_k4096": (1, 256, 129280, 4096, 8192, 4096), "longctx": (0, 4, 1048576, 512, 4096, 4096),
          "row65536": (1, 1, 65536, 512, 1024, 1024), "huge": (1, 1, 268435456, 32, 8192, 4096)}
print(json.dumps({n: ds.ds_get_plan(*a) for n, a in shapes.items()}))
"""


def test_plans_on_a_described_device(lib):
    """The planner's choices for the workload shapes, on a described 152-SM part with
    228 KB of shared memory per SM (no GPU needed): rows under 16 MB stay in one cluster
    (no merge pass), huge rows spread over clusters, one-CTA rows where k is large; where
    the CTAs are no more than the SMs (long-context and single rows), each CTA takes a
    whole SM's shared memory and holds all its chunks in a ring of up to 16 stages."""
    import json
    import sys
    env = dict(os.environ, DS_PLAN_DEVICE="152,232448,233472", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", _PLAN_SCRIPT], env=env, cwd=ROOT, capture_output=True,
                         text=True, check=True).stdout
    plans = json.loads(out.strip().splitlines()[-1])
    def pc(n):
        return plans[n]["parts"], plans[n]["cluster"], plans[n]["merge_launch"]
    assert pc("indexer") == (4, 4, 0)
    assert pc("sampler") == (1, 1, 0) and plans["sampler"]["threads"] == 256        # split-row kernel
    assert pc("sampler_k4096") == (1, 1, 0) and plans["sampler_k4096"]["threads"] == 256
    assert pc("longctx") == (16, 16, 0)
    assert pc("row65536") == (8, 8, 0)
    assert pc("huge") == (256, 8, 1)
    rows = {"indexer": 64, "sampler": 256, "sampler_k4096": 256, "longctx": 4, "row65536": 1, "huge": 1}
    for n, p in plans.items():
        assert p["smem_bytes"] <= 232448, n
        if p["threads"] == 256:
            assert p["stages"] in (8, 16), n          # warp-owned stages
            if rows[n] * p["parts"] <= 152:
                assert p["ctas_per_sm"] == 1 and p["chunk_elems"] * (2 if n in ("indexer", "longctx") else 4) <= 8192, n
            else:
                assert p["ctas_per_sm"] == 2, n


_PLAN_SWEEP = """
import json, top_selection_gb300 as ds
ds.load()
out = []
for dtype in (0, 1):
    for rows in (1, 3, 64, 256, 2048):
        for N in (1000, 4097, 65536, 131072, 1048576, 16777216):
            for k in (1, 64, 512, 2048, 4096):
                for B, B2 in ((1024, 1024), (4096, 4096), (8192, 4096)):
                    if k > N:
                        continue
                    try:
                        p = ds.ds_get_plan(dtype, rows, N, k, B, B2)
                    except Exception:
                        continue
                    out.append([dtype, rows, N, k, B, B2, p])
print(json.dumps(out))
"""


def test_split_plans_leave_a_chunk_of_room():
    """Every split-row plan over a sweep of shapes (no GPU needed) keeps a candidate buffer
    of at least k + one chunk: after a compaction to k a whole pass (at most one chunk of
    survivors) fits, which the compaction's progress rests on; the buffer also stays
    below 2^16 entries, the range of the final select's 16-bit bin counts."""
    import json
    import sys
    env = dict(os.environ, DS_PLAN_DEVICE="152,232448,233472", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", _PLAN_SWEEP], env=env, cwd=ROOT, capture_output=True,
                         text=True, check=True).stdout
    plans = json.loads(out.strip().splitlines()[-1])
    split = [r for r in plans if r[6]["threads"] == 256]
    assert len(split) > 100
    for dtype, rows, N, k, B, B2, p in split:
        es = 2 if dtype == 0 else 4
        assert p["capacity"] >= k + p["chunk_elems"], (dtype, rows, N, k, B, B2, p)
        assert p["capacity"] < 1 << 16, (dtype, rows, N, k, B, B2, p)
        assert (p["chunk_elems"] * es) % 16 == 0, (dtype, rows, N, k, B, B2, p)
        assert p["stages"] in (8, 16), (dtype, rows, N, k, B, B2, p)


def test_build_tracks_every_source_file():
    """Every CUDA source or header under csrc/ and every public header is a build input,
    so editing any of them makes the in-tree library out of date."""
    from top_selection_gb300 import build
    deps = set(build.deps())
    for d, exts in ((build.CSRC, (".cu", ".cuh", ".h")), (build.INCLUDE, (".h",))):
        for f in os.listdir(d):
            if f.endswith(exts):
                assert os.path.join(d, f) in deps, f


def test_touching_a_kernel_header_marks_the_library_stale(lib):
    from top_selection_gb300 import build
    assert build.up_to_date()
    split = os.path.join(build.CSRC, "ds_split.cuh")
    st = os.stat(split)
    try:
        t = os.path.getmtime(build.LIB) + 10
        os.utime(split, (t, t))
        assert not build.up_to_date()
    finally:
        os.utime(split, ns=(st.st_atime_ns, st.st_mtime_ns))
    assert build.up_to_date()


_BLOCKS_SCRIPT = r"""
import json, top_selection_gb300 as ds
ds.load()
out = {}
for rows in (1, 64, 152, 153, 256, 1000):
    p = ds.ds_get_plan(1, rows, 129280, 512, 0, 0)
    out[rows] = (p["B"], p["B2"])
q = ds.ds_get_plan(0, 64, 131072, 512, 4096, 0)
out["given_B"] = (q["B"], q["B2"])
q = ds.ds_get_plan(0, 64, 131072, 512, 0, 1024)
out["given_B2"] = (q["B"], q["B2"])
print(json.dumps(out))
"""


def test_library_chooses_block_sizes_on_a_described_device(lib):
    """B = 0 / B2 = 0: B is 8192 while the rows fit one wave of CTAs (rows <= SMs), 4096
    after that, B2 is 4096 (the shipped CUDA configuration the DeepSelect TopK tutorial
    describes, section 4.7); values passed explicitly are kept."""
    import json
    import sys
    env = dict(os.environ, DS_PLAN_DEVICE="152,232448,233472", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", _BLOCKS_SCRIPT], env=env, cwd=ROOT, capture_output=True,
                         text=True, check=True).stdout
    got = json.loads(out.strip().splitlines()[-1])
    for rows in ("1", "64", "152"):
        assert got[rows] == [8192, 4096]
    for rows in ("153", "256", "1000"):
        assert got[rows] == [4096, 4096]
    assert got["given_B"] == [4096, 4096]
    assert got["given_B2"] == [8192, 1024]


_SPEC_SCRIPT = r"""
import json, top_selection_gb300 as ds
ds.load()
out = {
    "indexer": ds.ds_get_plan(0, 64, 131072, 512, 4096, 4096),
    "indexer_k64": ds.ds_get_plan(0, 64, 131072, 64, 4096, 4096),
    "indexer_k2048": ds.ds_get_plan(0, 64, 131072, 2048, 4096, 4096),
    "longctx": ds.ds_get_plan(0, 4, 1048576, 512, 4096, 4096),
    "row65536": ds.ds_get_plan(1, 1, 65536, 512, 1024, 1024),
    "sampler": ds.ds_get_plan(1, 256, 129280, 512, 8192, 4096),
    "one_cta": ds.ds_get_plan(0, 64, 131072, 512, 4096, 4096, parts=1),
    "spread": ds.ds_get_plan(1, 1, 1 << 26, 512, 8192, 4096),
}
print(json.dumps(out))
"""


def test_speculative_rank_on_a_described_device(lib):
    """Rows held whole in one cluster speculate with spec_k = ceil(2 k S / N), S = the
    cluster's sampled elements (CTAs x two chunks x chunk), when 64 <= spec_k < k; rows
    streamed through the ring, rows over several clusters and the one-CTA schedule never
    do."""
    import json
    import sys
    env = dict(os.environ, DS_PLAN_DEVICE="152,232448,233472", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "-c", _SPEC_SCRIPT], env=env, cwd=ROOT, capture_output=True,
                         text=True, check=True).stdout
    got = json.loads(out.strip().splitlines()[-1])

    def expect(p, k, N):
        blocks = -(-(-(-N // p["B"])) // p["parts"])
        assert blocks * -(-p["B"] // p["chunk_elems"]) <= p["stages"]  # every chunk in the ring
        S = p["cluster"] * 2 * p["chunk_elems"]
        sk = -(-2 * k * S // N)
        return sk if 64 <= sk < k else 0

    assert got["indexer"]["spec_k"] == expect(got["indexer"], 512, 131072) == 256
    assert got["indexer_k64"]["spec_k"] == 0              # 32 < 64: too noisy
    assert got["indexer_k2048"]["spec_k"] == expect(got["indexer_k2048"], 2048, 131072) == 512
    assert got["row65536"]["spec_k"] == expect(got["row65536"], 512, 65536) == 256
    assert got["longctx"]["spec_k"] == expect(got["longctx"], 512, 1048576) == 128  # a whole SM per CTA: held
    assert got["sampler"]["spec_k"] == 0                   # streamed through the ring
    assert got["one_cta"]["spec_k"] == 0                   # the pages' one-CTA schedule
    assert got["spread"]["merge_launch"] == 1 and got["spread"]["spec_k"] == 0  # several clusters


def test_topk_sample_host_validation(lib):
    import top_selection_gb300 as ds
    a = [P, 1, 2, 1000, 1024, 8, 64, 64, 1]
    for t in (0.0, -1.0, float("nan"), float("inf")):
        assert ds.ds_topk_sample(*a, t, P, P, P, P, P, 0) == 1
    assert ds.ds_topk_sample(*a, 1.0, 0, P, P, P, P, 0) == 1      # no uniforms
    assert ds.ds_topk_sample(*a, 1.0, P, P, P, 0, P, 0) == 1      # no token output
    assert ds.ds_topk_sample(P, 1, 0, 1000, 1024, 8, 64, 64, 1, 1.0, 0, P, P, 0, 0, 0) == 0   # no rows
