"""The C-ABI boundary without a GPU: the library builds and loads, exports
every function include/detattn.h declares, and rejects invalid arguments with
the documented status codes before any CUDA call (so no device is needed)."""
import ctypes
import math

import numpy as np
import pytest

import deterministic_attention_gb300 as da


@pytest.fixture(scope="module")
def L():
    da.build()
    return da.lib()


def test_exports_every_declared_symbol(L):
    names = da.header_symbols()
    assert set(names) >= {"attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_bwd_delta",
                          "attn_bwd_dkdv", "attn_bwd_dq", "detattn_check_status",
                          "detattn_set_wait_limit_ns", "detattn_last_error", "detattn_version"}
    for n in names:
        assert hasattr(L, n), n


def test_dkdv_split_knob_validates(L):
    for ok in (0, 1, 2, 4, 8):
        assert L.detattn_set_dkdv_split(ok) == 0
    for bad in (-1, 3, 16):
        assert L.detattn_set_dkdv_split(bad) == -3
    assert L.detattn_set_dkdv_split(0) == 0


def test_version(L):
    assert L.detattn_version() == 10000


P = ctypes.c_void_p(0x10000)       # 16-byte aligned stand-in pointer (never dereferenced)
BAD = ctypes.c_void_p(0x10008)     # misaligned


def _fwd(L, q=P, k=P, v=P, o=P, lse=P, B=1, T=128, Hq=2, Hkv=1, D=64, scale=0.125, causal=1):
    return L.attn_fwd(q, k, v, o, lse, B, T, Hq, Hkv, D, scale, causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(lse=None), -1),
    (dict(v=BAD), -2), (dict(o=BAD), -2),
    (dict(B=-1), -3), (dict(T=-5), -3), (dict(Hq=3, Hkv=2), -3), (dict(Hkv=0), -3),
    (dict(D=96), -4), (dict(D=32), -4), (dict(D=256), -4),
    (dict(scale=0.0), -5), (dict(scale=-1.0), -5), (dict(scale=math.inf), -5),
    (dict(scale=math.nan), -5), (dict(causal=2), -5),
])
def test_fwd_rejects(L, kw, code):
    assert _fwd(L, **kw) == code
    assert da.last_error() != ""


def test_empty_problem_is_ok_without_device(L):
    assert _fwd(L, q=None, k=None, v=None, o=None, lse=None, B=0) == 0
    assert _fwd(L, T=0, q=None) == 0


def test_workspace_bytes(L):
    # Row statistics rounded up to 256 bytes, then 256 bytes for the dQ step's
    # tile counter.
    assert L.attn_bwd_workspace_bytes(4, 1024, 12, 4, 64) == 4 * 12 * 1024 * 8 + 256
    assert L.attn_bwd_workspace_bytes(1, 3, 1, 1, 64) == 128 * 8 + 256
    assert L.attn_bwd_workspace_bytes(2, 129, 3, 1, 128) == 2 * 3 * 256 * 8 + 256
    assert L.attn_bwd_workspace_bytes(1, 1, 1, 1, 64) == 1024 + 256
    assert L.attn_bwd_workspace_bytes(1, 3, 3, 2, 64) == 0
    assert L.attn_bwd_workspace_bytes(0, 3, 2, 1, 64) == 0


def test_bwd_rejects(L):
    args = [P] * 10
    def call(ws=P, wsb=1 << 20, **kw):
        a = dict(B=1, T=128, Hq=2, Hkv=1, D=64, scale=0.125, causal=1)
        a.update(kw)
        v = list(args)
        v[9] = ws
        return L.attn_bwd(*v, wsb, a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["scale"],
                          a["causal"], None)
    assert call(ws=None) == -9
    assert call(wsb=100) == -9
    assert call(ws=BAD) == -2
    assert call(D=80) == -4
    assert call(Hq=5, Hkv=2) == -3
    assert L.attn_bwd_dq(P, P, P, P, P, 1 << 20, None, 1, 128, 2, 1, 64, 0.125, 1, None) == -1
    assert L.attn_bwd_dq(P, P, P, P, P, 100, P, 1, 128, 2, 1, 64, 0.125, 1, None) == -9
    assert L.attn_bwd_dkdv(P, P, P, P, P, 1 << 20, P, BAD, 1, 128, 2, 1, 64, 0.125, 1, None) == -2
    assert L.attn_bwd_dkdv(P, P, P, P, None, 1 << 20, P, P, 1, 128, 2, 1, 64, 0.125, 1, None) == -9
    assert L.attn_bwd_delta(P, P, None, P, 1 << 20, 1, 128, 2, 64, None) == -1
    assert L.attn_bwd_delta(P, P, P, BAD, 1 << 20, 1, 128, 2, 64, None) == -2


def test_python_binding_refuses_cpu_tensors(L):
    import torch
    q = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        da.attn_fwd(q, q[:, :, :1], q[:, :, :1])


@pytest.mark.parametrize("D,B,T,Hq,causal,sms", [
    (64, 4, 1024, 12, 1, 152),    # page3: the host's listed deal
    (64, 32, 1024, 24, 1, 152),   # past the list: rounds dealt in alternating directions
    (128, 1, 8192, 32, 1, 152),   # one pipeline per block, past the list
    (64, 1, 512, 12, 1, 152),     # fewer units than SMs
    (64, 2, 300, 3, 0, 8),        # full attention on few SMs
    (128, 3, 1000, 5, 1, 132),
])
def test_qtile_deal(D, B, T, Hq, causal, sms):
    """The dQ step's static deal of 128-query tiles to its blocks (one
    pipeline each; host logic, no GPU): every unit goes to exactly one
    pipeline, and no pipeline's load exceeds the mean by more than one unit;
    past the host list (1,024 units) the deal is round k of the pipelines,
    forward in even rounds, backward in odd.  A unit weighs its 128-key tiles
    plus two."""
    n_pipes, pipe = da.diag_qtile_deal(D, B, T, Hq, causal, sms)
    n_m = -(-T // 128)
    units = B * Hq * n_m
    assert n_pipes == min(sms, units)
    assert pipe.shape == (units,) and (pipe >= 0).all() and (pipe < n_pipes).all()
    kv = -(-T // 128)
    mt = n_m - 1 - np.arange(units) // (B * Hq)
    n_kv = np.minimum(kv, (mt * 128 + 128) // 128) if causal else np.full(units, kv)
    w = n_kv + 2.0
    load = np.bincount(pipe, weights=w, minlength=n_pipes)
    assert load.max() <= w.sum() / n_pipes + w.max()
    if units > 1024:
        k, i = np.divmod(np.arange(units), n_pipes)
        assert (pipe == np.where(k % 2 == 0, i, n_pipes - 1 - i)).all()


def test_qtile_deal_validates():
    with pytest.raises(da.DetAttnError):
        da.diag_qtile_deal(96, 1, 128, 2, 1, 152)  # head dim
    with pytest.raises(da.DetAttnError):
        da.diag_qtile_deal(64, 1, 128, 2, 1, 0)    # no SMs
    assert da.diag_qtile_deal(64, 0, 128, 2, 1, 152)[0] == 0


# A GB300-like device for the split model: 152 SMs, one dK/dV block per SM,
# clusters placed without loss (152 / C of them).  Nominal, not queried.
_RESIDENT = [152, 76, 38, 19]


def test_dkdv_split_picks_the_measured_best():
    """The cost model's automatic C at the three D = 64 shapes whose C was
    measured on a GB300 at every value (fastest: C = 4 at 1x512x12/4,
    C = 2 at 4x1024x12/4, C = 1 at 32x1024x24/24), and NG = min(key tiles,
    resident clusters of that C)."""
    assert da.diag_dkdv_split(1, 512, 12, 4, 64, True, _RESIDENT) == (4, 16)
    assert da.diag_dkdv_split(4, 1024, 12, 4, 64, True, _RESIDENT) == (2, 76)
    assert da.diag_dkdv_split(32, 1024, 24, 24, 64, True, _RESIDENT) == (1, 152)
    # D = 128, 1x8192x32/8: one block per tile (the 128-query kernel, tiles
    # heaviest first) measured 1.00 ms against 1.44 ms with C = 2.
    assert da.diag_dkdv_split(1, 8192, 32, 8, 128, True, _RESIDENT) == (1, 152)


@pytest.mark.parametrize("shape", [(1, 128, 2, 1, 64), (4, 1024, 12, 4, 64),
                                   (1, 8192, 32, 8, 128), (3, 777, 6, 2, 128)])
def test_dkdv_split_invariants(shape):
    B, T, Hq, Hkv, D = shape
    tiles = B * Hkv * -(-T // 128)
    limit = 8 if D == 64 else 2
    c, ng = da.diag_dkdv_split(*shape, True, _RESIDENT)
    assert c in (1, 2, 4, 8) and c <= limit
    assert ng == min(tiles, _RESIDENT[c.bit_length() - 1])
    for forced in (1, 2, 4, 8):
        fc, fng = da.diag_dkdv_split(*shape, True, _RESIDENT, forced)
        assert fc == min(forced, limit)
        assert fng == min(tiles, _RESIDENT[fc.bit_length() - 1])
    # A cluster size the device cannot hold is never chosen.
    res = list(_RESIDENT)
    res[c.bit_length() - 1] = 0
    if any(res[: limit.bit_length()]):
        assert da.diag_dkdv_split(*shape, True, res)[0] != c


def test_dkdv_split_validates():
    assert da.diag_dkdv_split(0, 128, 2, 1, 64, True, _RESIDENT) == (0, 0)
    with pytest.raises(da.DetAttnError):
        da.diag_dkdv_split(1, 128, 2, 1, 64, True, [0, 0, 0, 0])  # nothing resident
    with pytest.raises(da.DetAttnError):
        da.diag_dkdv_split(1, 128, 2, 1, 64, True, _RESIDENT, 3)  # not a power of two
    with pytest.raises(da.DetAttnError):
        da.diag_dkdv_split(1, 128, 3, 2, 64, True, _RESIDENT)     # Hq % Hkv
    # D = 64 allows clusters of 8; at D = 128 a forced 8 acts as 2, which this
    # device cannot hold.
    assert da.diag_dkdv_split(1, 128, 2, 1, 64, True, [0, 0, 0, 5], 8) == (8, 1)
    with pytest.raises(da.DetAttnError):
        da.diag_dkdv_split(1, 128, 2, 1, 128, True, [152, 0, 0, 5], 8)


def _check_dkdv_list(lists, B, T, Hq, Hkv, c, ng):
    """Every key tile is dealt once: whole to one block, or shared by all c
    blocks of one cluster, which list it among their shared tiles in the
    same order; each block's shared tiles come first."""
    n_tiles = B * Hkv * -(-T // 128)
    assert len(lists) == c * ng
    seen = {}
    for i, lst in enumerate(lists):
        flags = [sh for _, sh in lst]
        assert flags == sorted(flags, reverse=True), f"block {i}: shared tiles not first"
        for t, sh in lst:
            assert 0 <= t < n_tiles
            seen.setdefault(t, []).append((i, sh))
    assert sorted(seen) == list(range(n_tiles))
    for t, holders in seen.items():
        if holders[0][1]:
            blocks = sorted(i for i, _ in holders)
            assert all(sh for _, sh in holders) and len(blocks) == c
            assert blocks == list(range(blocks[0], blocks[0] + c)) and blocks[0] % c == 0
        else:
            assert len(holders) == 1
    for g in range(ng):
        shared = [[t for t, sh in lists[g * c + j] if sh] for j in range(c)]
        assert all(x == shared[0] for x in shared), f"cluster {g}: peers disagree"


def test_dkdv_list_at_page3():
    """At 4x1024x12/4 (C = 2 over 76 clusters) the automatic deal lists the
    tiles: the three heaviest tile rows (24, 21, 18 items) shared, the rest
    whole, so no block waits on a peer for a light tile."""
    lists = da.diag_dkdv_list(4, 1024, 12, 4, True, 2, 76)
    assert lists is not None
    _check_dkdv_list(lists, 4, 1024, 12, 4, 2, 76)
    BH = 4 * 4
    for lst in lists:
        for t, sh in lst:
            assert sh == (t // BH < 3), (t, sh)
    assert max(len(lst) for lst in lists) == 2


@pytest.mark.parametrize("shape,c,ng", [((2, 520, 6, 2), 2, 3), ((1, 1024, 3, 1), 4, 2),
                                        ((6, 1024, 3, 1), 8, 19), ((24, 1024, 3, 1), 2, 76),
                                        ((3, 700, 8, 2), 2, 76)])
def test_dkdv_list_invariants(shape, c, ng):
    forced = da.diag_dkdv_list(*shape, True, c, ng, force=True)
    assert forced is not None
    _check_dkdv_list(forced, *shape, c, ng)
    auto = da.diag_dkdv_list(*shape, True, c, ng)
    if auto is not None:
        assert auto == forced
    assert da.diag_dkdv_list(*shape, False, c, ng, force=True) is not None


def test_dkdv_list_validates():
    assert da.diag_dkdv_list(0, 128, 2, 1, True, 2, 1) is None
    for c, ng in ((1, 4), (3, 4), (16, 1), (2, 0)):
        with pytest.raises(da.DetAttnError):
            da.diag_dkdv_list(1, 1024, 2, 1, True, c, ng)
    # More blocks than a list holds: the plain walk.
    assert da.diag_dkdv_list(64, 1024, 2, 2, True, 2, 200, force=True) is None
    da.set_dkdv_deal(0)
    with pytest.raises(da.DetAttnError):
        da.set_dkdv_deal(3)


def test_size_limits_reject_before_any_device_call(L):
    """Shapes beyond the kernels' index limits fail validation (no device is
    needed to reach the answer)."""
    assert _fwd(L, B=1 << 20, T=1 << 20, Hq=16, Hkv=1) == -3     # elements > 1e12
    assert _fwd(L, B=1, T=(1 << 30) + 1, Hq=1, Hkv=1) == -3      # T > 2^30
    assert "too large" in da.last_error()
    assert L.attn_bwd_workspace_bytes(1 << 20, 1 << 20, 16, 1, 64) == 0


def _has_gpu():
    import torch
    return torch.cuda.is_available()


def test_noalloc_rejects(L):
    def call(B=1, T=128, Hq=2, Hkv=1, D=64, ptr=P, scale=0.125):
        return L.attn_bwd_noalloc(P, P, P, P, P, P, ptr, P, P, B, T, Hq, Hkv, D, scale, 1, None)
    # B * Hq * Tp row-statistic pairs above the built-in 2^20: a workspace error.
    assert call(B=4, T=1024, Hq=257) == -9                 # 4 * 257 * 1024 > 2^20
    assert "exceeds the built-in scratch" in da.last_error()
    assert call(B=16, T=1025, Hq=64, Hkv=8) == -9         # Tp = 1152: 1,179,648 pairs
    if not _has_gpu():
        # Just under the limit validation passes, and only the missing device
        # stops the call.  (Never made where a GPU exists: the pointers here
        # are stand-ins.)
        assert call(B=8, T=1025, Hq=64, Hkv=8) == -6
    assert call(ptr=None) == -1
    assert call(ptr=BAD) == -2
    assert call(D=96) == -4
    assert call(scale=0.0) == -5
    assert call(B=0, ptr=None) == 0                       # empty: nothing to do


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every call raises: there is no fallback."""
    monkeypatch.setattr(da, "_lib", None)
    monkeypatch.setattr(da, "_LIB_PATH", str(tmp_path / "libdetattn.so"))
    with pytest.raises(RuntimeError, match="not built"):
        da.lib()
    with pytest.raises(RuntimeError, match="not built"):
        da.last_error()


def test_product_shares_nothing_with_the_oracle():
    """The package (binding, build, kernels, host layer) never imports,
    includes or links the oracle; only tests, smoke and the bench's CPU legs do."""
    import glob
    import os
    pkg = os.path.dirname(da.__file__)
    files = (glob.glob(os.path.join(pkg, "*.py")) + glob.glob(os.path.join(pkg, "csrc", "*")) +
             glob.glob(os.path.join(os.path.dirname(pkg), "include", "*")))
    assert len(files) >= 8
    for f in files:
        text = open(f, errors="replace").read()
        for needle in ("import oracle", "from oracle", "attn_oracle", "embed_oracle", "liboracle"):
            assert needle not in text, (f, needle)


# Threads that share one SM's 65,536 registers for each kernel: its block size
# times the blocks it keeps per SM.
_KERNEL_THREADS_PER_SM = {
    "attn_fwd_kernelILi64E": 384, "attn_fwd_kernelILi128E": 256,
    "attn_dq_kernelILi64E": 384, "attn_dq_kernelILi128E": 384,
    "attn_dkdvq_kernelILi64E": 384, "attn_dkdvq_kernelILi128E": 384,
    "attn_dkdv_kernelILi128E": 608,
    "attn_delta_kernelILi64E": 4 * 256, "attn_delta_kernelILi128E": 4 * 256,
}


def _ptxas_entries():
    """(kernel, registers, spill store bytes, spill load bytes) from the
    build's ptxas reports."""
    import importlib
    import re
    b = importlib.import_module("deterministic_attention_gb300.build")
    out = []
    for src in b.SOURCES:
        text = open(b.resource_report_path(src)).read()
        for chunk in text.split("Compiling entry function '")[1:]:
            name = chunk.split("'", 1)[0]
            regs = int(re.search(r"Used (\d+) registers", chunk).group(1))
            sp = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", chunk)
            out.append((name, regs, int(sp.group(1)), int(sp.group(2))))
    return out


# Spill stores (bytes) a kernel may keep.  The 64-dim forward runs two
# pipelines in 384 threads and moves registers from its control warpgroup
# (TMA producers, MMA issuers) to the softmax warpgroups, whose threads hold
# a row of 128 scores each; the control warps' issue loops keep a few values
# in local memory.
_SPILL_ALLOWANCE = {"attn_fwd_kernelILi64E": 64}
# Registers the 64-dim forward's warpgroups hold after reallocation: 128
# control threads at 56 and 256 softmax threads at 208.
_FWD64_REG_BUDGET = 128 * 56 + 256 * 208


def test_kernels_fit_their_launch_without_spills(L):
    entries = _ptxas_entries()
    seen = set()
    for name, regs, st, ld in entries:
        allowed = max([v for k, v in _SPILL_ALLOWANCE.items() if k in name], default=0)
        assert st <= allowed, f"{name} spills {st}/{ld} bytes"
        if "attn_fwd_kernelILi64E" in name:
            # The softmax warpgroups' increase must be covered by the
            # registers the block launches with.
            assert regs * 384 >= _FWD64_REG_BUDGET, f"{name}: {regs} registers at launch"
        for key, threads in _KERNEL_THREADS_PER_SM.items():
            if key in name:
                seen.add(key)
                assert regs * threads <= 65536, f"{name}: {regs} registers x {threads} threads"
    assert seen == set(_KERNEL_THREADS_PER_SM), f"kernels not found in the reports: {seen}"


def test_embed_grad_rejects_before_any_device_call(L):
    """embed_grad validates shapes, pointers and the workspace on the host."""
    def call(N=64, V=100, E=128, ids=P, dy=P, dw=P, ws=P, wsb=1 << 30):
        return L.embed_grad(ids, dy, dw, ws, wsb, N, V, E, None)
    assert call(N=-1) == -3
    assert call(V=0) == -3
    assert call(E=6) == -3                       # not a multiple of 4
    assert call(E=0) == -3
    assert call(ids=None) == -1
    assert call(dw=None) == -1
    assert call(ws=None) == -1
    assert call(dy=BAD) == -2
    assert call(wsb=16) == -9
    assert "workspace needs" in da.last_error()
    assert L.embed_grad_workspace_bytes(-1, 5, 8) == 0
    # counts, offsets, cursor (V, V + 1, V ints), two token lists (N ints) and
    # two partial-row blocks of ceil(N / 32) x E floats, each 256-aligned.
    up = lambda x: (x + 255) // 256 * 256
    N, V, E = 1000, 50432, 1536
    want = (up(4 * V) + up(4 * (V + 1)) + up(4 * V) + 2 * up(4 * N)
            + 2 * up(4 * ((N + 31) // 32) * E))
    assert L.embed_grad_workspace_bytes(N, V, E) == want
    if not _has_gpu():
        assert call() == -6                     # valid: only the missing device stops it
        assert call(N=0, ids=None, dy=None) == -6


def test_varlen_rejects_before_any_device_call(L):
    """attn_fwd_varlen / attn_bwd_varlen validate the host offsets first."""
    def fwd(cu_q, cu_k, n_seq=None, Hq=4, Hkv=2, D=64, ptr=P):
        cq = np.asarray(cu_q, dtype=np.int32)
        ck = np.asarray(cu_k, dtype=np.int32)
        n = len(cq) - 1 if n_seq is None else n_seq
        return L.attn_fwd_varlen(P, P, P, ptr, P, ctypes.c_void_p(cq.ctypes.data),
                                 ctypes.c_void_p(ck.ctypes.data), n, Hq, Hkv, D, 0.125, 1, None)
    assert fwd([1, 5], [0, 5]) == -3                 # does not start at 0
    assert fwd([0, 5, 3], [0, 5, 9]) == -3           # decreases
    assert fwd([0, 5], [0, 5], n_seq=257) == -3      # too many sequences
    assert fwd([0, 5], [0, 5], Hq=3) == -3
    assert fwd([0, 5], [0, 5], D=32) == -4
    assert fwd([0, 5], [0, 5], ptr=None) == -1
    assert fwd([0, 0, 0], [0, 4, 9]) == 0            # no query rows: nothing to do
    # More than 2048 query tiles of 128 rows over the batch: 9 x 65,536 rows.
    big = [65536 * i for i in range(10)]
    assert fwd(big, big) == -3
    assert "tiles" in da.last_error()
    assert L.attn_bwd_varlen_workspace_bytes(None, None, 1, 4, 2, 64) == 0
    cq = np.asarray([0, 100, 300], dtype=np.int32)
    ws = L.attn_bwd_varlen_workspace_bytes(ctypes.c_void_p(cq.ctypes.data),
                                           ctypes.c_void_p(cq.ctypes.data), 2, 4, 2, 64)
    # Row statistics: Hq * (128 + 256) pairs of 8 bytes, rounded to 256, + 256.
    assert ws == (4 * 384 * 8 + 255) // 256 * 256 + 256
    if not _has_gpu():
        assert fwd([0, 100, 300], [0, 100, 300]) == -6


def test_layer_calls_reject_before_any_device_call(L):
    def gemm(M=128, N=128, K=64, lda=64, ldb=128, ldc=128, a=P, a_mn=0, b_mn=1, c_f32=0):
        return L.layer_gemm(a, a_mn, lda, P, b_mn, ldb, P, c_f32, ldc, M, N, K, 1.0, None)
    assert gemm(M=100) == -3
    assert gemm(N=96) == -3
    assert gemm(K=32) == -3
    assert gemm(lda=32) == -3           # shorter than K
    assert gemm(ldc=100) == -3
    assert gemm(a=None) == -1
    assert gemm(a=BAD) == -2
    assert gemm(a_mn=2) == -3
    assert L.layer_workspace_bytes(4, 1024, 768, 12, 4, 64) > 0
    assert L.layer_workspace_bytes(4, 1000, 768, 12, 4, 64) == 0   # B*T not a multiple of 128
    assert L.layer_workspace_bytes(4, 1024, 700, 12, 4, 64) == 0
    if not _has_gpu():
        assert gemm() == -6
