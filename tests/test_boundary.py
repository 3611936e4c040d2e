"""Host-side tests of the C ABI (no GPU needed).

The library must load, export every function include/attn.h declares, and
reject bad arguments with the documented status before touching the device,
with a message naming the offending field (as the page's validate_config does:
oxicuda-dnn 0.1.8 hopper.rs, validate_config and its tests).
"""

import ctypes
import os
import re

import pytest

from exact_attention_53_gb300 import binding
from exact_attention_53_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

A = 1 << 20          # a fake, 16-byte aligned "device" address; never dereferenced
MB = 1 << 24


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[a-z_][\w \*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert names == sorted(["attn_fwd", "attn_fwd_general", "attn_fwd_host", "attn_fwd_plan", "attn_fwd_splitkv_plan",
                            "attn_fwd_splitkv", "attn_fwd_splitkv_noalloc", "attn_bwd_workspace_size",
                            "attn_bwd", "attn_bwd_general", "attn_fwd_splitkv_general_plan",
                            "attn_fwd_splitkv_general", "attn_last_error", "attn_get_device_status",
                            "attn_version"])


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    probe = open(os.path.join(ROOT, "include", "attn_probe.h")).read()
    for name in binding.PROBES:
        assert re.search(rf"\b{name}\s*\(", probe) and hasattr(lib, name), name
    assert set(binding.EXPORTED) == set(_declared_functions())
    assert lib.attn_version() == 10000


def test_debug_library_exports_only_its_hooks(lib):
    """The failure-detection hooks live in libattn_debug.so alone, as include/attn_debug.h
    declares; the release library exports none of them."""
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "attn_debug.h")).read(),
                  flags=re.S)
    declared = sorted(set(re.findall(r"\b(attn_debug_\w+)\s*\(", text)))
    assert declared == sorted(binding.DEBUG_EXPORTS)
    dbg = binding.load_debug_library()
    for name in declared:
        assert hasattr(dbg, name), name
        assert not hasattr(lib, name), name


def _exported(path):
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if not nm:
        pytest.skip("nm is not installed")
    out = subprocess.run([nm, "-D", "--defined-only", path], stdout=subprocess.PIPE, text=True,
                         check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_libraries_export_only_their_c_abi(lib):
    """Each library exports the functions its headers declare and nothing else of its own, so
    loading both in one process never mixes their template code or its static state."""
    pkg = os.path.dirname(binding.library_path())
    ours = {n for n in _exported(binding.library_path()) if n.startswith("attn")}
    assert ours == set(_declared_functions()) | set(binding.PROBES)
    assert not {n for n in _exported(binding.library_path()) if "attn" in n and n not in ours}
    dbg = _exported(os.path.join(pkg, "libattn_debug.so"))
    assert {n for n in dbg if "attn" in n} == set(binding.DEBUG_EXPORTS)


def test_debug_entry_rejects_bad_arguments_before_device_work():
    dbg = binding.load_debug_library()
    assert dbg.attn_debug_fwd(None, A, A, A, A, 1, 1, 128, 0.125, -1, 0, None) == 1
    assert dbg.attn_debug_fwd(A, A, A, A, A, 1, 1, 0, 0.125, -1, 0, None) == 1
    assert dbg.attn_debug_bwd(None, *[A] * 9, 1, 1, 128, 0.125, -1, 0, None) == 1
    assert dbg.attn_debug_bwd(*[A] * 9, None, 1, 1, 128, 0.125, -1, 0, None) == 1
    assert dbg.attn_debug_bwd(*[A] * 10, 1, 1, 0, 0.125, -1, 0, None) == 1
    assert dbg.attn_debug_status(None, None) == 1


def _fwd(lib, q=A, k=A + MB, v=A + 2 * MB, o=A + 3 * MB, lse=A + 4 * MB, B=1, H=2, S_q=128,
         S_k=128, d=128, causal=0, scale=0.125, dtype=1):
    return lib.attn_fwd(q, k, v, o, lse, B, H, S_q, S_k, d, causal, scale, dtype, None)


CASES = [
    (dict(q=0), binding.ATTN_ERR_INVALID_ARG, "q is null"),
    (dict(k=0), binding.ATTN_ERR_INVALID_ARG, "k is null"),
    (dict(v=0), binding.ATTN_ERR_INVALID_ARG, "v is null"),
    (dict(o=0), binding.ATTN_ERR_INVALID_ARG, "o is null"),
    (dict(lse=0), binding.ATTN_ERR_INVALID_ARG, "lse is null"),
    (dict(B=0), binding.ATTN_ERR_INVALID_ARG, "B must be"),
    (dict(H=-1), binding.ATTN_ERR_INVALID_ARG, "H must be"),
    (dict(S_q=0), binding.ATTN_ERR_INVALID_ARG, "S_q must be"),
    (dict(S_k=0), binding.ATTN_ERR_INVALID_ARG, "S_k must be"),
    (dict(d=0), binding.ATTN_ERR_INVALID_ARG, "d must be"),
    (dict(d=96), binding.ATTN_ERR_UNSUPPORTED, "head_dim"),
    (dict(d=512), binding.ATTN_ERR_UNSUPPORTED, "head_dim"),
    (dict(dtype=2), binding.ATTN_ERR_UNSUPPORTED, "dtype"),
    (dict(causal=2), binding.ATTN_ERR_INVALID_ARG, "causal"),
    (dict(scale=float("nan")), binding.ATTN_ERR_INVALID_ARG, "scale"),
    (dict(scale=float("inf")), binding.ATTN_ERR_INVALID_ARG, "scale"),
    (dict(q=A + 8), binding.ATTN_ERR_INVALID_ARG, "q is not 16-byte aligned"),
    (dict(k=A + MB + 2), binding.ATTN_ERR_INVALID_ARG, "k is not 16-byte aligned"),
    (dict(o=A + 3 * MB + 4), binding.ATTN_ERR_INVALID_ARG, "o is not 16-byte aligned"),
    (dict(lse=A + 4 * MB + 2), binding.ATTN_ERR_INVALID_ARG, "lse is not 4-byte aligned"),
    (dict(o=A + 64), binding.ATTN_ERR_INVALID_ARG, "o overlaps q"),
    (dict(lse=A + 2 * MB + 16), binding.ATTN_ERR_INVALID_ARG, "lse overlaps v"),
    (dict(lse=A + 3 * MB + 1024), binding.ATTN_ERR_INVALID_ARG, "lse overlaps o"),
    (dict(S_q=(1 << 22) + 1), binding.ATTN_ERR_INVALID_ARG, "S_q"),
    (dict(S_k=(1 << 22) + 1, k=A + 8 * MB, v=A + 16 * MB * 256), binding.ATTN_ERR_INVALID_ARG, "S_k"),
    (dict(B=1 << 16, H=1 << 16), binding.ATTN_ERR_INVALID_ARG, "B*H"),
]


@pytest.mark.parametrize("kw,status,msg", CASES, ids=[c[2] for c in CASES])
def test_validation_rejects_before_device_work(lib, kw, status, msg):
    assert _fwd(lib, **kw) == status
    assert msg in lib.attn_last_error().decode()


def test_negative_scale_passes_validation(lib):
    """Any finite scale is accepted (the page's sm_scale is a plain f32): a negative one gets
    past validation to the device check, which fails here without a GPU."""
    assert _fwd(lib, scale=-0.5) == binding.ATTN_ERR_CUDA
    assert "scale" not in lib.attn_last_error().decode()


def test_host_entry_point_checks_host_pointers(lib):
    dev = [A, A + MB, A + 2 * MB, A + 3 * MB, A + 4 * MB]
    host = [A + 10 * MB, A + 11 * MB, A + 12 * MB, A + 13 * MB, A + 14 * MB]
    for i, name in enumerate(["q_host", "k_host", "v_host", "o_host", "lse_host"]):
        h = list(host)
        h[i] = 0
        st = lib.attn_fwd_host(*h, *dev, 1, 2, 128, 128, 128, 0, 0.125, 1, None)
        assert st == binding.ATTN_ERR_INVALID_ARG
        assert name in lib.attn_last_error().decode()
    d2 = list(dev)
    d2[1] = A + 64          # k_dev overlapping q_dev
    st = lib.attn_fwd_host(*host, *d2, 1, 2, 128, 128, 128, 0, 0.125, 1, None)
    assert st == binding.ATTN_ERR_INVALID_ARG


def test_valid_call_without_gpu_reports_cuda_error(lib):
    """With no usable device, a valid call fails cleanly with ATTN_ERR_CUDA/UNSUPPORTED."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _fwd(lib)
    assert st in (binding.ATTN_ERR_CUDA, binding.ATTN_ERR_UNSUPPORTED)
    assert lib.attn_last_error().decode()


def test_python_wrapper_raises_on_bad_input(lib):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float32)
    with pytest.raises(binding.AttnError):
        binding.fwd(q, q, q)
    with pytest.raises(binding.AttnError):
        binding.fwd(q[0], q[0], q[0])


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setenv("ATTN_LIBRARY", str(tmp_path / "nope.so"))
    with pytest.raises(binding.AttnError, match="missing"):
        binding.load_library()
    monkeypatch.setattr(binding, "_lib", None)


GOLDEN = os.path.join(ROOT, "tests", "golden", "launch_grid_cases.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(tuple(int(x) for x in line.split()))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: "x".join(map(str, r)))
def test_plan_matches_page_launch_grid(lib, row):
    """The query-tile count and head count agree with the page's launch_params cases."""
    S_q, S_k, B, H, q_tiles, bh = row
    for d in (64, 128):
        plan = binding.attn_fwd_plan(B, H, S_q, S_k, d, 0, binding.ATTN_DTYPE_F16)
        assert plan.block_m == 128
        assert plan.q_tiles == q_tiles
        assert plan.bh == bh
        assert plan.units == bh * -(-q_tiles // plan.q_tiles_per_cta)


def test_plan_resources_fit_the_sm():
    build()
    for d in (64, 128, 256):
        for causal in (0, 1):
            p = binding.attn_fwd_plan(2, 3, 1000, 700, d, causal, binding.ATTN_DTYPE_BF16)
            assert p.smem_bytes <= 232448
            assert p.tmem_cols <= 512
            assert p.threads % 128 == 0
            assert p.kv_tiles == 6 and p.q_tiles == 8
            assert p.q_tiles_per_cta == (1 if d == 256 else 2)


def test_plan_validates_like_fwd(lib):
    with pytest.raises(binding.AttnError, match="head_dim"):
        binding.attn_fwd_plan(1, 1, 16, 16, 80, 0, binding.ATTN_DTYPE_BF16)
    with pytest.raises(binding.AttnError, match="S_q must be"):
        binding.attn_fwd_plan(1, 1, 0, 16, 64, 0, binding.ATTN_DTYPE_BF16)
    assert lib.attn_fwd_plan(1, 1, 16, 16, 64, 0, 1, None) == binding.ATTN_ERR_INVALID_ARG


# ------------------------------------------------------------------ split-KV


@pytest.mark.parametrize("S_k,n_req,n_used", [
    (128, 4, 1),            # one key tile: one range whatever is asked
    (1000, 1, 1),
    (1000, 3, 3),           # 8 tiles -> 3,3,2
    (1000, 5, 4),           # 8 tiles: ceil(8/5)=2 per range -> 4 ranges, none empty
    (1000, 8, 8),
    (1000, 50, 8),          # capped at the tile count
    (16384, 7, 7),          # 128 tiles: 19 per range -> 7 ranges
    (16385, 128, 65),       # 129 tiles: 2 per range -> 65 ranges
])
def test_splitkv_plan_ranges_and_workspace(lib, S_k, n_req, n_used):
    B, H, S_q, d = 2, 3, 37, 128
    n, ws = binding.attn_fwd_splitkv_plan(B, H, S_q, S_k, d, binding.ATTN_DTYPE_BF16, n_req)
    assert n == n_used
    assert ws == (n * B * H * S_q * (d + 1) * 4 if n > 1 else 0)
    tiles = -(-S_k // 128)
    per = -(-tiles // n)
    assert (n - 1) * per < tiles <= n * per      # every range holds at least one tile


def _split(lib, q=A, k=A + MB, v=A + 2 * MB, o=A + 3 * MB, lse=A + 4 * MB, B=1, H=2, S_q=16,
           S_k=4096, d=128, scale=0.125, dtype=1, n_split=4, ws=A + 8 * MB, ws_bytes=1 << 22):
    return lib.attn_fwd_splitkv(q, k, v, o, lse, B, H, S_q, S_k, d, scale, dtype, n_split, ws,
                                ws_bytes, None)


SPLIT_CASES = [
    (dict(n_split=-1), binding.ATTN_ERR_INVALID_ARG, "n_split must be"),
    (dict(ws=0), binding.ATTN_ERR_INVALID_ARG, "workspace is null"),
    (dict(ws=A + 8 * MB + 8), binding.ATTN_ERR_INVALID_ARG, "workspace is not 16-byte aligned"),
    (dict(ws_bytes=4 * 2 * 16 * 129 * 4 - 1), binding.ATTN_ERR_INVALID_ARG, "workspace_bytes"),
    (dict(ws=A + 64), binding.ATTN_ERR_INVALID_ARG, "workspace overlaps q"),
    (dict(ws=A + 3 * MB), binding.ATTN_ERR_INVALID_ARG, "workspace overlaps o"),
    (dict(ws=A + 4 * MB - 1024), binding.ATTN_ERR_INVALID_ARG, "workspace overlaps lse"),
    (dict(d=96), binding.ATTN_ERR_UNSUPPORTED, "head_dim"),
    (dict(q=0), binding.ATTN_ERR_INVALID_ARG, "q is null"),
    (dict(o=A + 64), binding.ATTN_ERR_INVALID_ARG, "o overlaps q"),
]


@pytest.mark.parametrize("kw,status,msg", SPLIT_CASES, ids=[c[2] for c in SPLIT_CASES])
def test_splitkv_validation_rejects_before_device_work(lib, kw, status, msg):
    assert _split(lib, **kw) == status
    assert msg in lib.attn_last_error().decode()


def test_splitkv_plan_validates(lib):
    with pytest.raises(binding.AttnError, match="n_split must be"):
        binding.attn_fwd_splitkv_plan(1, 1, 16, 4096, 128, binding.ATTN_DTYPE_BF16, -2)
    with pytest.raises(binding.AttnError, match="head_dim"):
        binding.attn_fwd_splitkv_plan(1, 1, 16, 4096, 80, binding.ATTN_DTYPE_BF16, 2)
    n = ctypes.c_int64()
    assert lib.attn_fwd_splitkv_plan(1, 1, 16, 16, 64, 1, 1, None, ctypes.byref(n)) == \
        binding.ATTN_ERR_INVALID_ARG


def test_noalloc_rejects_plans_above_the_built_in_scratch(lib):
    """64 ranges of 4·32·256·129·4 bytes exceed the 16 MiB scratch: rejected on the host."""
    B, H, S_q, S_k, d = 4, 32, 256, 16384, 128
    n, ws = binding.attn_fwd_splitkv_plan(B, H, S_q, S_k, d, binding.ATTN_DTYPE_BF16, 64)
    assert ws > binding.NOALLOC_SCRATCH_BYTES
    st = lib.attn_fwd_splitkv_noalloc(A, A + (1 << 30), A + (2 << 30), A + (3 << 30),
                                      A + (4 << 30), B, H, S_q, S_k, d, 0.125, 1, 64, None)
    assert st == binding.ATTN_ERR_INVALID_ARG
    msg = lib.attn_last_error().decode()
    assert "scratch" in msg and str(binding.NOALLOC_SCRATCH_BYTES) in msg


def test_noalloc_header_states_the_scratch_size():
    text = open(HEADER).read()
    m = re.search(r"#define ATTN_NOALLOC_SCRATCH_BYTES \((\d+) \* 1024 \* 1024\)", text)
    assert m and int(m.group(1)) * 1024 * 1024 == binding.NOALLOC_SCRATCH_BYTES


# ------------------------------------------------------------------ backward


def test_bwd_workspace_size(lib):
    assert binding.attn_bwd_workspace_size(2, 3, 300, 77, 128, binding.ATTN_DTYPE_BF16) == \
        2 * 6 * 384 * 4
    assert binding.attn_bwd_workspace_size(1, 1, 128, 1, 64, binding.ATTN_DTYPE_F16) == 2 * 128 * 4
    assert binding.attn_bwd_workspace_size(1, 1, 129, 128, 256, binding.ATTN_DTYPE_BF16) == \
        2 * 256 * 4
    with pytest.raises(binding.AttnError, match="head_dim"):
        binding.attn_bwd_workspace_size(1, 1, 128, 128, 96, binding.ATTN_DTYPE_BF16)


def _bwd(lib, **kw):
    G = 1 << 24
    args = dict(q=A, k=A + G, v=A + 2 * G, o=A + 3 * G, lse=A + 4 * G, dout=A + 5 * G,
                dq=A + 6 * G, dk=A + 7 * G, dv=A + 8 * G, B=1, H=2, S_q=256, S_k=256, d=128,
                causal=0, scale=0.125, dtype=1, ws=A + 9 * G, ws_bytes=1 << 20)
    args.update(kw)
    a = args
    return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dout"], a["dq"], a["dk"],
                        a["dv"], a["B"], a["H"], a["S_q"], a["S_k"], a["d"], a["causal"],
                        a["scale"], a["dtype"], a["ws"], a["ws_bytes"], None)


BWD_CASES = [
    (dict(d=96), binding.ATTN_ERR_UNSUPPORTED, "head_dim"),
    (dict(dout=0), binding.ATTN_ERR_INVALID_ARG, "dout is null"),
    (dict(dq=0), binding.ATTN_ERR_INVALID_ARG, "dq is null"),
    (dict(ws=0), binding.ATTN_ERR_INVALID_ARG, "workspace is null"),
    (dict(dk=A + (7 << 24) + 8), binding.ATTN_ERR_INVALID_ARG, "dk is not 16-byte aligned"),
    (dict(lse=A + (4 << 24) + 2), binding.ATTN_ERR_INVALID_ARG, "lse is not 4-byte aligned"),
    (dict(ws_bytes=2 * 2 * 256 * 4 - 1), binding.ATTN_ERR_INVALID_ARG, "workspace_bytes"),
    (dict(dq=A + 64), binding.ATTN_ERR_INVALID_ARG, "dq overlaps q"),
    (dict(dv=A + (7 << 24) + 1024), binding.ATTN_ERR_INVALID_ARG, "dk overlaps dv"),
    (dict(ws=A + (8 << 24)), binding.ATTN_ERR_INVALID_ARG, "overlaps"),
    (dict(causal=3), binding.ATTN_ERR_INVALID_ARG, "causal"),
]


@pytest.mark.parametrize("kw,status,msg", BWD_CASES, ids=[c[2] for c in BWD_CASES])
def test_bwd_validation_rejects_before_device_work(lib, kw, status, msg):
    assert _bwd(lib, **kw) == status
    assert msg in lib.attn_last_error().decode()


# ------------------------------------------------------------------ general layouts


def _gen(lib, **kw):
    G = 1 << 28
    B, H, H_kv, S_q, S_k, d = kw.pop("B", 2), kw.pop("H", 4), kw.pop("H_kv", 2), kw.pop("S_q", 64), \
        kw.pop("S_k", 96), kw.pop("d", 64)
    dense = lambda heads, S: binding.AttnLayout(heads * S * d, S * d, d)  # noqa: E731
    p = binding.AttnFwdParams(A, A + G, A + 2 * G, A + 3 * G, A + 4 * G, B, H, H_kv, S_q, S_k, d,
                              dense(H, S_q), dense(H_kv, S_k), dense(H_kv, S_k), dense(H, S_q),
                              1, 0.125, 1)
    for key, val in kw.items():
        setattr(p, key, val)
    return lib.attn_fwd_general(ctypes.byref(p), None)


GEN_CASES = [
    (dict(H_kv=3), binding.ATTN_ERR_INVALID_ARG, "H_kv=3 must divide H=4"),
    (dict(H_kv=0), binding.ATTN_ERR_INVALID_ARG, "H_kv=0"),
    (dict(mask=5), binding.ATTN_ERR_INVALID_ARG, "mask must be"),
    (dict(mask=2, S_q=200, S_k=100), binding.ATTN_ERR_UNSUPPORTED, "S_q <= S_k"),
    (dict(q_layout=binding.AttnLayout(8 * 64 * 64, 64 * 64, 60)), binding.ATTN_ERR_INVALID_ARG,
     "q row stride 60"),
    (dict(k_layout=binding.AttnLayout(0, 96 * 64, 64)), binding.ATTN_ERR_INVALID_ARG, "k batch stride"),
    (dict(o_layout=binding.AttnLayout(64 * 64, 64, 64)), binding.ATTN_ERR_INVALID_ARG,
     "o layout maps two elements"),
    (dict(o=A + (1 << 28) + 4096), binding.ATTN_ERR_INVALID_ARG, "o overlaps k"),
    (dict(d=128, q_layout=binding.AttnLayout(4 * 64 * 128, 64 * 128, 64)), binding.ATTN_ERR_INVALID_ARG,
     "below d=128"),
]


@pytest.mark.parametrize("kw,status,msg", GEN_CASES, ids=[c[2] for c in GEN_CASES])
def test_general_validation(lib, kw, status, msg):
    assert _gen(lib, **kw) == status
    assert msg in lib.attn_last_error().decode()


def test_general_accepts_packed_and_head_major_views(lib):
    """BSHD views of one packed [B, S, 3, H, d] buffer pass validation (then fail only for lack of a GPU)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    B, H, S, d = 2, 4, 64, 64
    packed = binding.AttnLayout(S * 3 * H * d, d, 3 * H * d)
    st = _gen(lib, B=B, H=H, H_kv=H, S_q=S, S_k=S, d=d, q_layout=packed, k_layout=packed,
              v_layout=packed, k=A + H * d * 2, v=A + 2 * H * d * 2,
              o_layout=binding.AttnLayout(S * H * d, d, H * d))
    assert st in (binding.ATTN_ERR_CUDA, binding.ATTN_ERR_UNSUPPORTED)


def test_splitkv_general_plan_and_mask_rules(lib):
    G = 1 << 28
    d = 128
    dense = lambda heads, S: binding.AttnLayout(heads * S * d, S * d, d)  # noqa: E731
    p = binding.AttnFwdParams(A, A + G, A + 2 * G, A + 3 * G, A + 4 * G, 2, 32, 8, 1, 9000, d,
                              dense(32, 1), dense(8, 9000), dense(8, 9000), dense(32, 1), 0, 0.1, 1)
    n, ws = binding.attn_fwd_splitkv_general_plan(p, 6)
    assert n == 6 and ws == 6 * 2 * 32 * 1 * (d + 1) * 4
    p.mask = binding.ATTN_MASK_CAUSAL_BOTTOM_RIGHT          # one query row: same as full
    assert binding.attn_fwd_splitkv_general_plan(p, 6)[0] == 6
    p.mask = binding.ATTN_MASK_CAUSAL
    with pytest.raises(binding.AttnError, match="full attention"):
        binding.attn_fwd_splitkv_general_plan(p, 6)


def test_resource_report_strips_parameter_lists():
    from exact_attention_53_gb300.build import _strip_params
    assert (_strip_params("void attn::attn_fwd_kernel<(int)128, (bool)1>(CUtensorMap_st, int)")
            == "attn::attn_fwd_kernel<(int)128, (bool)1>")
    assert _strip_params("<unnamed>::ex2_rate_kernel(float*, int)") == "<unnamed>::ex2_rate_kernel"


@pytest.mark.parametrize("lang", ["c99", "c++17"])
def test_public_headers_compile_as_plain_c_and_cpp(tmp_path, lang):
    """include/*.h is a C ABI: it must compile on its own as strict C99 and as C++, with no
    CUDA or torch headers on the include path."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c99" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    headers = sorted(f for f in os.listdir(inc) if f.endswith(".h"))
    src = tmp_path / "use_headers.c"
    src.write_text("".join(f'#include "{h}"\n' for h in headers) + "int main(void) { return 0; }\n")
    cmd = [cc, f"-std={lang}", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I", inc]
    if lang == "c99":
        cmd.append("-pedantic")
    else:
        cmd += ["-x", "c++"]
    r = subprocess.run(cmd + [str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
