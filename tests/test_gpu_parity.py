"""CUDA path vs the oracle, through the C ABI, on the five seeded workloads.

Small and scaled sizes are compared element by element on every call; the full
sizes (124M, the 1.196e9 decoder bucket, 1.07e9 with statistics) are compared
on sampled indices, which is exact because elements are independent, and the
statistics against the oracle's sum over the whole gradient.
"""

import dataclasses

import numpy as np
import pytest
import torch

import amsgrad_optimizer_step_gb300 as fa
from gpu_harness import run_workload
from synthetic.configs import (CONFIG1, CONFIG2, CONFIG3, CONFIG4, CONFIG4_MAX, CONFIG5,
                               decoder_bucket_shapes)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from amsgrad_optimizer_step_gb300 import build
    build.build()
    torch.cuda.init()


def sample_indices(n, k=40000, seed=0, extra=()):
    rng = np.random.default_rng(seed)
    base = set(rng.integers(0, n, k).tolist())
    for b in (0, 1, 2, 7, 8, 9, 4095, 4096, 4097, n - 9, n - 8, n - 7, n - 2, n - 1, *extra):
        if 0 <= b < n:
            base.add(int(b))
    return np.array(sorted(base), dtype=np.int64)


def small_decoder_offsets(scale=32):
    sizes = []
    for _, shape in decoder_bucket_shapes()[:1 + 9 * 3]:  # embed + 3 layers
        sizes.append(int(np.prod([max(1, d // scale) for d in shape])))
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


# ---- the five workloads ---------------------------------------------------------

def test_config1_out_of_place_full():
    s = run_workload(CONFIG1, CONFIG1.n, "oop", DEV, guard=1024)
    assert s["updates"] == 10 and s["t"] == 10


def test_config2_bf16_scaled_amsgrad_with_skip_full():
    s = run_workload(CONFIG2, CONFIG2.n, "oop", DEV, guard=1024)
    assert s["skips"] == 1 and s["updates"] == 19 and s["t"] == 19


@pytest.mark.parametrize("api", ["inplace", "oop"])
def test_config3_scaled_ragged(api):
    w = dataclasses.replace(CONFIG3, calls=12, inplace=api == "inplace")
    s = run_workload(w, 1_000_003, api, DEV, guard=1024)
    assert s["t"] == 12


def test_config3_full_size_sampled():
    idx = sample_indices(CONFIG3.n, seed=3)
    s = run_workload(CONFIG3, CONFIG3.n, "inplace", DEV, idx=idx)
    assert s["t"] == 50


@pytest.mark.parametrize("w", [CONFIG4, CONFIG4_MAX], ids=["maximize_off", "maximize_on"])
def test_config4_scaled_decoder_bucket(w):
    off = small_decoder_offsets()
    s = run_workload(w, int(off[-1]), "bucket", DEV, segments=off, guard=1024)
    assert s["t"] == 10


@pytest.mark.parametrize("w", [CONFIG4, CONFIG4_MAX], ids=["maximize_off", "maximize_on"])
def test_config4_full_size_sampled(w):
    idx = sample_indices(w.n, seed=4, extra=list(w.segments[1:-1]) + [x - 1 for x in w.segments[1:-1]])
    s = run_workload(w, w.n, "bucket", DEV, idx=idx)
    assert s["t"] == 10


@pytest.mark.parametrize("api", ["clipped", "gated"])
def test_config5_scaled_stats_clip_and_inf_skip(api):
    n = 256 * 5000 + 77
    s = run_workload(CONFIG5, n, api, DEV, row_len=256, guard=1024)
    assert s["skips"] == 1 and s["updates"] == 4 and s["t"] == 4
    # norm well above 1: the clip is active in every update
    assert all(r[1] > 1.0 for r in s["reports"] if r[3] == 0)


def test_config5_full_size_sampled():
    idx = sample_indices(CONFIG5.n, seed=5, extra=[CONFIG5.inf_index()])
    s = run_workload(CONFIG5, CONFIG5.n, "clipped", DEV, idx=idx, row_len=256,
                     full_grad_on_host=False)
    assert s["skips"] == 1 and s["t"] == 4
    inf_reports = [r for r in s["reports"] if r[3] > 0]
    assert len(inf_reports) == 1 and inf_reports[0][2] == 1


# ---- sizes, dtypes, alignment ---------------------------------------------------

@pytest.mark.parametrize("gdt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("ams", [False, True])
@pytest.mark.parametrize("n", [1, 2, 7, 8, 9, 15, 16, 17, 255, 4095, 4097, 65537])
def test_edge_sizes(gdt, ams, n):
    w = dataclasses.replace(CONFIG1, grad_dtype=gdt, amsgrad=ams, calls=3, inplace=True)
    run_workload(w, n, "inplace", DEV, guard=64)


@pytest.mark.parametrize("gdt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("offsets", [(1, 1, 1, 1, 1), (3, 3, 3, 3, 3), (0, 1, 2, 3, 5),
                                     (2, 0, 0, 0, 0), (0, 0, 0, 0, 3)])
def test_misaligned_views(gdt, offsets):
    """Views starting off a 16-byte boundary: common offset -> vector body after a
    scalar head; mixed offsets -> all-scalar kernel.  Both must match the oracle."""
    n = 10_001
    w = dataclasses.replace(CONFIG2, grad_dtype=gdt, calls=3, skip_calls=(), amsgrad=True,
                            inplace=True).scaled(n)
    import oracle
    lib = oracle.lib()
    idx = np.arange(n)
    bufs = []
    names = ("p", "m", "v", "vmax")
    views = {}
    for name, off in zip(names, offsets[:4]):
        full = torch.zeros(n + 16, dtype=torch.float32, device=DEV)
        bufs.append(full)
        views[name] = full[off:off + n]
    gfull = torch.zeros(n + 16, dtype={"f32": torch.float32, "f16": torch.float16,
                                       "bf16": torch.bfloat16}[gdt], device=DEV)
    g = gfull[offsets[4]:offsets[4] + n]
    w.fill_params_device(views["p"])
    traj = oracle.OracleAdamW(w.params_host(idx), w.options(), lib_=lib)
    t = 0
    for call in range(1, 4):
        w.fill_grad_device(call, g)
        t, upd = fa.fa_adamw_step_inplace(views["p"], g, views["m"], views["v"], views["vmax"], t,
                                          fa.options(**w.options()),
                                          fa.control(w.gradient_scale))
        traj.step(w.grad_host(call, idx), gdt, w.gradient_scale)
    torch.cuda.synchronize()
    from gpu_harness import gate
    gate(views["p"].cpu().numpy(), traj.p, 1e-6, "p")
    gate(views["vmax"].cpu().numpy(), traj.state.vmax, 1e-6, "vmax")


@pytest.mark.parametrize("api", ["clipped", "gated"])
def test_more_than_2_31_elements_sampled(api):
    """A bucket of 2^31 + 777 parameters (8.6 GB per FP32 array): every element offset in
    the kernels is 64-bit; the norm matches the oracle's over the whole gradient, and
    sampled elements on both sides of 2^31, at the ragged end and at random match it too,
    first step and steady steps, with the update decided on the host and on the device."""
    n = 2 ** 31 + 777
    w = dataclasses.replace(CONFIG3, calls=3, inplace=True, outlier_per_10000=0,
                            max_grad_norm=1.0, row_len=1024)
    edges = [2 ** 31 - 9, 2 ** 31 - 1, 2 ** 31, 2 ** 31 + 1, 2 ** 31 + 8, 2 ** 30 * 3 // 2]
    idx = sample_indices(n, k=20000, seed=31, extra=edges)
    # the whole statistics-guarded step: analysis in rows of 1024 (2,097,153 rows), the
    # merge, the norm against the oracle's sum over all 2^31 + 777 values, the clipped update
    s = run_workload(w, n, api, DEV, idx=idx, row_len=1024, full_grad_on_host=False)
    assert s["t"] == 3 and s["updates"] == 3
    assert all(r[1] > 1.0 for r in s["reports"])  # the clip is active


def _random_case(k):
    rng = np.random.default_rng(1000 + k)
    n = int(rng.choice([1, 7, 4097, 65_537, 300_001, 1_000_003, 3_000_017]))
    scale = float(2.0 ** rng.integers(-2, 8))
    return dataclasses.replace(
        CONFIG2, name=f"random{k}", seed=int(rng.integers(1, 10_000)),
        grad_dtype=str(rng.choice(["f32", "f16", "bf16"])), amsgrad=bool(rng.integers(2)),
        maximize=bool(rng.integers(2)), lr=float(10 ** rng.uniform(-5, -1)),
        beta1=float(rng.choice([0.0, 0.5, 0.9, 0.95])),
        beta2=float(rng.choice([0.9, 0.99, 0.999, 0.9999])),
        eps=float(10 ** rng.uniform(-10, -3)), weight_decay=float(rng.choice([0.0, 1e-4, 0.1])),
        gradient_scale=scale, grad_premul=scale, calls=int(rng.integers(2, 5)),
        skip_calls=(2,) if rng.integers(3) == 0 else (), inplace=True).scaled(n)


@pytest.mark.parametrize("k", range(24))
def test_random_configurations_vs_oracle(k):
    """Seeded random combinations of size, gradient dtype, AMSGrad, maximize, lr, betas,
    eps, decay, power-of-two loss scale, call count and an occasional skip, each against
    the oracle (one step from identical state and along the trajectory)."""
    w = _random_case(k)
    s = run_workload(w, w.n, "inplace", DEV, guard=64)
    assert s["t"] == w.calls - len(w.skip_calls)


# ---- degenerate hyper-parameters ------------------------------------------------

DEGENERATE = {
    "lr0": dict(lr=0.0),
    "wd0": dict(weight_decay=0.0),
    "beta1_0": dict(beta1=0.0),
    "beta2_0": dict(beta2=0.0),
    "betas_0": dict(beta1=0.0, beta2=0.0),
    # seed 4: no gradient value is exactly zero at these sizes (with eps 0 a zero
    # gradient on the first step gives 0/0 on both sides)
    "eps0": dict(eps=0.0, seed=4),
}


@pytest.mark.parametrize("n", [4097, 1_000_003])
@pytest.mark.parametrize("name", sorted(DEGENERATE))
def test_degenerate_options_vs_oracle(name, n):
    """Boundary values of the options: lr 0 (p must stay bit-identical), no decay,
    beta1 or beta2 = 0 (bias corrections exactly 1), eps 0 (no zero gradient present)."""
    w = dataclasses.replace(CONFIG2, calls=4, skip_calls=(), amsgrad=True, inplace=True,
                            **DEGENERATE[name]).scaled(n)
    if name == "eps0":
        for call in range(1, w.calls + 1):
            assert not (widen(w, call) == 0).any(), "a zero gradient would make 0/0 here"
    p0 = None
    if name == "lr0":
        p0 = torch.empty(n, device=DEV)
        w.fill_params_device(p0)
    s = run_workload(w, n, "inplace", DEV, guard=64)
    assert s["t"] == 4
    if p0 is not None:
        assert torch.equal(s["state"].p, p0)


def widen(w, call):
    from gpu_harness import widen_host
    return widen_host(w.grad_host(call, np.arange(w.n)), w.grad_dtype)


@pytest.mark.parametrize("t", [1_000, 1_000_000, 100_000_000])
def test_large_step_count_vs_oracle(t, oracle_lib):
    """Far into training beta^t underflows and the bias corrections are exactly 1."""
    from gpu_harness import gate, oracle_one_step
    n = 100_003
    w = dataclasses.replace(CONFIG2, amsgrad=True, skip_calls=()).scaled(n)
    opts = w.options()
    p, m, v, vm = (torch.empty(n, device=DEV) for _ in range(4))
    w.fill_params_device(p)
    rng = np.random.default_rng(11)
    for x in (m, v, vm):
        x.copy_(torch.from_numpy(rng.random(n, dtype=np.float32) * 1e-4))
    vm.copy_(torch.maximum(vm, v))
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    w.fill_grad_device(1, g)
    before = [x.double().cpu().numpy() for x in (p, m, v, vm)]
    t_new, upd = fa.fa_adamw_step_inplace(p, g, m, v, vm, t, fa.options(**opts),
                                          fa.control(w.gradient_scale))
    torch.cuda.synchronize()
    assert t_new == t + 1 and upd
    ref = oracle_one_step(w.grad_host(1, np.arange(n)), w.grad_dtype, opts, w.gradient_scale,
                          1.0, t + 1, before, oracle_lib)
    for dev_x, ref_x, nm in zip((p, m, v, vm), ref, "p m v vmax".split()):
        gate(dev_x.cpu().numpy(), ref_x, 1e-6, f"t={t} {nm}")


@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_non_finite_gradients_propagate_like_the_oracle(gdt, oracle_lib):
    """A plain step takes no finiteness decision: NaN and +-Inf in the gradient follow
    IEEE arithmetic, and the AMSGrad max keeps a NaN once it has one.  Special values must
    sit exactly where the oracle has them; everything else within the usual tolerance."""
    import oracle
    n = 1_000_003  # steady steps take the shared-memory pipeline
    w = dataclasses.replace(CONFIG2, grad_dtype=gdt, calls=3, skip_calls=(), amsgrad=True,
                            inplace=True, gradient_scale=1.0, grad_premul=1.0).scaled(n)
    opts = w.options()
    idx = np.arange(n)
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p)
    m, v, vm = (torch.zeros(n, device=DEV) for _ in range(3))
    g = torch.empty(n, dtype={"f32": torch.float32, "bf16": torch.bfloat16}[gdt], device=DEV)
    ref = oracle.OracleAdamW(w.params_host(idx), opts, lib_=oracle_lib)
    planted = {1: {5: float("nan"), 77_777: float("inf")},
               2: {5: 1.0, 123_456: float("-inf"), 999_999: float("nan")},
               3: {}}
    t = 0
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        for i, x in planted[call].items():
            g[i] = x
        from gpu_harness import grad_bits_from_device
        bits = grad_bits_from_device(g)
        t, _ = fa.fa_adamw_step_inplace(p, g, m, v, vm, t, fa.options(**opts), fa.control())
        ref.step(bits, gdt)
        torch.cuda.synchronize()
        for dev_x, ref_x, nm in ((p, ref.p, "p"), (m, ref.state.m, "m"), (v, ref.state.v, "v"),
                                 (vm, ref.state.vmax, "vmax")):
            d = dev_x.cpu().numpy().astype(np.float64)
            r = np.asarray(ref_x, np.float64)
            assert np.array_equal(np.isnan(d), np.isnan(r)), f"call {call} {nm}: NaN positions"
            assert np.array_equal(np.isposinf(d), np.isposinf(r)), f"call {call} {nm}: +Inf"
            assert np.array_equal(np.isneginf(d), np.isneginf(r)), f"call {call} {nm}: -Inf"
            fin = np.isfinite(r)
            from gpu_harness import gate
            gate(d[fin], r[fin], 1e-5, f"call {call} {nm} (finite elements)")
    assert np.isnan(vm[5].item()), "the AMSGrad max keeps the NaN of call 1"


# ---- bitwise invariants ---------------------------------------------------------

def _fresh(n, gdt, seed, ams=True):
    w = dataclasses.replace(CONFIG2, grad_dtype=gdt, amsgrad=ams, seed=seed, skip_calls=(),
                            inplace=True, gradient_scale=1.0, grad_premul=1.0)
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p) if n == w.n else w.scaled(n).fill_params_device(p)
    return w if n == w.n else w.scaled(n), p


def _grads(w, call):
    g = torch.empty(w.n, dtype={"f32": torch.float32, "f16": torch.float16,
                                "bf16": torch.bfloat16}[w.grad_dtype], device=DEV)
    w.fill_grad_device(call, g)
    return g


def _zeros(n, k):
    return [torch.zeros(n, device=DEV) for _ in range(k)]


@pytest.mark.parametrize("gdt", ["f32", "bf16", "f16"])
def test_inplace_equals_out_of_place_bitwise(gdt):
    w, p0 = _fresh(70_001, gdt, 11)
    o = fa.options(**w.options())
    pa = p0.clone()
    ma, va, vma = _zeros(w.n, 3)
    pb, mb, vb, vmb, tb = p0.clone(), None, None, None, 0
    ta = 0
    for call in range(1, 6):
        g = _grads(w, call)
        ta, _ = fa.fa_adamw_step_inplace(pa, g, ma, va, vma, ta, o, fa.control())
        pb, mb, vb, vmb, tb, _ = fa.fa_adamw_step(pb, g, mb, vb, vmb, tb, o, fa.control())
    torch.cuda.synchronize()
    assert ta == tb == 5
    for a, b in ((pa, pb), (ma, mb), (va, vb), (vma, vmb)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_bucket_equals_per_tensor_bitwise():
    off = small_decoder_offsets(16)
    n = int(off[-1])
    w, p0 = _fresh(n, "f16", 12)
    o = fa.options(**w.options())
    pa, pb = p0.clone(), p0.clone()
    ma, va, vma = _zeros(n, 3)
    mb, vb, vmb = _zeros(n, 3)
    ta = 0
    tb = [0] * (len(off) - 1)
    for call in range(1, 4):
        g = _grads(w, call)
        ta, _ = fa.fa_bucket_step(list(off), pa, g, ma, va, vma, ta, o, fa.control())
        for k in range(len(off) - 1):
            s = slice(int(off[k]), int(off[k + 1]))
            tb[k], _ = fa.fa_adamw_step_inplace(pb[s], g[s], mb[s], vb[s], vmb[s], tb[k], o,
                                                fa.control())
    torch.cuda.synchronize()
    for a, b in ((pa, pb), (ma, mb), (va, vb), (vma, vmb)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_maximize_equals_negated_gradient_bitwise(gdt):
    w, p0 = _fresh(33_333, gdt, 13)
    pa, pb = p0.clone(), p0.clone()
    sa, sb = _zeros(w.n, 3), _zeros(w.n, 3)
    ta = tb = 0
    oa = fa.options(**dict(w.options(), maximize=True))
    ob = fa.options(**dict(w.options(), maximize=False))
    for call in range(1, 4):
        g = _grads(w, call)
        gneg = g.clone()
        if gdt == "f32":
            gneg.neg_()
        else:
            gneg.view(torch.int16).bitwise_xor_(torch.tensor(-32768, dtype=torch.int16, device=DEV))
        ta, _ = fa.fa_adamw_step_inplace(pa, g, *sa, ta, oa, fa.control())
        tb, _ = fa.fa_adamw_step_inplace(pb, gneg, *sb, tb, ob, fa.control())
    torch.cuda.synchronize()
    assert torch.equal(pa, pb) and all(torch.equal(x, y) for x, y in zip(sa, sb))
    assert not torch.equal(pa, p0)


def test_power_of_two_scale_bitwise():
    w, p0 = _fresh(20_000, "bf16", 14)
    pa, pb = p0.clone(), p0.clone()
    sa, sb = _zeros(w.n, 3), _zeros(w.n, 3)
    o = fa.options(**w.options())
    ta = tb = 0
    for call in range(1, 4):
        g = _grads(w, call)
        g128 = (g.float() * 128).to(torch.bfloat16)  # exact: power of two, no overflow
        ta, _ = fa.fa_adamw_step_inplace(pa, g, *sa, ta, o, fa.control(1.0))
        tb, _ = fa.fa_adamw_step_inplace(pb, g128, *sb, tb, o, fa.control(128.0))
    torch.cuda.synchronize()
    assert torch.equal(pa, pb) and all(torch.equal(x, y) for x, y in zip(sa, sb))


def test_checkpoint_export_import_bitwise():
    """10 straight steps == 5 steps, export state, restore into fresh buffers, 5 steps."""
    w, p0 = _fresh(50_001, "f16", 15)
    o = fa.options(**w.options())
    grads = [_grads(w, c) for c in range(1, 11)]
    pa = p0.clone()
    sa = _zeros(w.n, 3)
    ta = 0
    for g in grads:
        ta, _ = fa.fa_adamw_step_inplace(pa, g, *sa, ta, o, fa.control())
    pb = p0.clone()
    sb = _zeros(w.n, 3)
    tb = 0
    for g in grads[:5]:
        tb, _ = fa.fa_adamw_step_inplace(pb, g, *sb, tb, o, fa.control())
    torch.cuda.synchronize()
    saved = {"t": tb, "p": pb.cpu(), "m": sb[0].cpu(), "v": sb[1].cpu(), "vmax": sb[2].cpu()}
    del pb, sb
    pc = saved["p"].to(DEV)
    sc = [saved[k].to(DEV) for k in ("m", "v", "vmax")]
    tc = saved["t"]
    for g in grads[5:]:
        tc, _ = fa.fa_adamw_step_inplace(pc, g, *sc, tc, o, fa.control())
    torch.cuda.synchronize()
    assert ta == tc == 10
    assert torch.equal(pa, pc) and all(torch.equal(x, y) for x, y in zip(sa, sc))


def test_skip_and_empty_launch_nothing():
    w, p0 = _fresh(1000, "f32", 16)
    o = fa.options(**w.options())
    g = _grads(w, 1)
    # out of place, skip: returns the very same tensors, allocates nothing
    before = torch.cuda.memory_allocated()
    p2, m2, v2, vm2, t2, upd = fa.fa_adamw_step(p0, g, None, None, None, 0, o,
                                                fa.control(skip_update=True))
    assert p2 is p0 and m2 is None and t2 == 0 and not upd
    assert torch.cuda.memory_allocated() == before
    e = torch.empty(0, device=DEV)
    p3, _, _, _, t3, upd3 = fa.fa_adamw_step(e, e, None, None, None, 4, o, fa.control())
    assert t3 == 4 and not upd3


# ---- statistics kernels ---------------------------------------------------------

def grad_bits(t):
    """Storage bits of a device gradient on the host: float32 values, or uint16 patterns."""
    t = t.cpu()
    return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)


def _planted_grad(n, gdt, seed, bad_idx, sigma=1e-2):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(n) * sigma).astype(np.float32)
    vals = [np.inf, -np.inf, np.nan]
    for j, i in enumerate(bad_idx):
        x[i] = vals[j % 3]
    t = torch.from_numpy(x)
    t = t.to({"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[gdt])
    bits = t.numpy() if gdt == "f32" else t.view(torch.int16).numpy().view(np.uint16)
    return t.to(DEV), bits


@pytest.mark.parametrize("gdt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("n,row_len,segs", [
    (256 * 1000, 256, None), (256 * 777 + 5, 256, None), (12_345, 100, None), (3, 256, None),
    (100_000, 256, [0, 1, 2049, 70_000, 70_000, 100_000]), (65_536, 7, None)])
def test_analyze_rows_match_oracle(gdt, n, row_len, segs, oracle_lib):
    bad = [0, n // 3, n - 1] if n > 3 else [1]
    g, bits = _planted_grad(n, gdt, 21, bad)
    rows = fa.fa_stats_rows(n, row_len, segs)
    buf = fa.stats_buffer(rows, DEV)
    got = fa.fa_analyze_gradient(g, row_len, buf, segs)
    torch.cuda.synchronize()
    assert got == rows
    rs, rc = oracle_lib.row_stats(bits, gdt, row_len, segs)
    host = buf.cpu()
    dev_s = host[:rows, 0].view(torch.float32).double().numpy()
    dev_c = host[:rows, 1].numpy().astype(np.int64)
    dev_lo = host[:rows, 2].view(torch.float32).double().numpy()
    assert np.array_equal(dev_c, rc.astype(np.int64))
    ok = rc == 0
    assert np.all(np.abs(dev_s + dev_lo - rs)[ok] <= 2e-6 * rs[ok] + 1e-30)


def _decoded_records(host, rows):
    """Sums of squares of the first ``rows`` records: plain ones added here, scaled ones
    (negative first word) decoded by the library."""
    hi = host[:rows, 0].view(torch.float32).double().numpy()
    lo = host[:rows, 2].view(torch.float32).double().numpy()
    out = hi + lo
    for r in np.flatnonzero(hi < 0):
        rec = fa.FaStats()
        rec.sum_sq, rec.nonfinite, rec.sum_sq_lo = float(hi[r]), int(host[r, 1]), float(lo[r])
        out[r] = fa.fa_stats_sum_sq(rec)
    return out


@pytest.mark.parametrize("k", range(16))
def test_random_statistics_vs_oracle(k, oracle_lib):
    """Seeded random analyses: size, gradient dtype, row length (fast and generic kernels),
    segment tables with empty segments, 0-5 planted NaN/+-Inf values and, in FP32 and BF16
    cases, 0-3 finite values whose squares overflow FP32.  Every row record against the
    oracle (counts exact), then the merged report (count exact, sum within the merge's
    error) and the skip / clip decision."""
    import math
    rng = np.random.default_rng(5000 + k)
    gdt = str(rng.choice(["f32", "f16", "bf16"]))
    n = int(rng.integers(1, 2_000_000))
    row_len = int(rng.choice([1, 7, 100, 256, 512, 1000, 1024, 2048]))
    segs = None
    if rng.integers(2):
        cuts = np.sort(rng.integers(0, n + 1, int(rng.integers(1, 40))))
        segs = [0] + [int(x) for x in cuts] + [n]
    rows = fa.fa_stats_rows(n, row_len, segs)
    if rows > 4_194_304:
        row_len, rows = 1024, fa.fa_stats_rows(n, 1024, segs)
    bad = [int(i) for i in rng.integers(0, n, int(rng.integers(0, 6)))]
    g, bits = _planted_grad(n, gdt, 6000 + k, bad)
    if gdt != "f16":  # finite values beyond sqrt(FP32 max); FP16's largest squares fit
        huge = [(int(i), float(v)) for i, v in zip(rng.integers(0, n, int(rng.integers(0, 4))),
                                                   10.0 ** rng.uniform(19.5, 38.4, 4))
                if int(i) not in bad]
        for i, val in huge:
            g[i] = val
        bits = grad_bits(g)
    buf = fa.stats_buffer(rows, DEV)
    assert fa.fa_analyze_gradient(g, row_len, buf, segs) == rows
    scratch = fa.scratch_buffer(rows, DEV)
    report = fa.stats_buffer(1, DEV)
    fa.fa_merge_gradient_stats(buf, rows, scratch, report)
    torch.cuda.synchronize()
    rs, rc = oracle_lib.row_stats(bits, gdt, row_len, segs)
    host = buf.cpu()
    dev_c = host[:rows, 1].numpy().astype(np.int64)
    dev_sum = _decoded_records(host, rows)
    assert np.array_equal(dev_c, rc.astype(np.int64))
    ok = rc == 0
    assert np.all(np.abs(dev_sum - rs)[ok] <= 2e-6 * rs[ok] + 1e-30)
    h = fa.fa_read_report(report)
    s_or, c_or = oracle_lib.gradient_stats(bits, gdt)
    assert h.nonfinite == c_or
    if c_or == 0:
        got = fa.fa_stats_sum_sq(h)
        exact_rows = math.fsum(dev_sum.tolist())
        assert abs(got - exact_rows) <= 1e-12 * exact_rows
        assert abs(got - s_or) <= 2e-6 * s_or + 1e-30


@pytest.mark.parametrize("rows", [1, 2, 1023, 1024, 1025, 4096, 1_048_575, 1_048_576,
                                  1_048_577, 4_194_304])
def test_merge_matches_exact_sum(rows):
    """The merge only reorders the sum: compare with math.fsum of the records."""
    import math
    rng = np.random.default_rng(rows)
    s = (rng.random(rows) * 10).astype(np.float32)
    lo = (rng.random(rows) * 1e-7).astype(np.float32)
    c = rng.integers(0, 3, rows).astype(np.int32) * (rng.random(rows) < 1e-3)
    host = torch.zeros((rows, 3), dtype=torch.int32)
    host[:, 0] = torch.from_numpy(s).view(torch.int32)
    host[:, 1] = torch.from_numpy(c.astype(np.int32))
    host[:, 2] = torch.from_numpy(lo).view(torch.int32)
    rows_in = host.to(DEV)
    scratch = fa.scratch_buffer(rows, DEV)
    report = fa.stats_buffer(1, DEV)
    fa.fa_merge_gradient_stats(rows_in, rows, scratch, report)
    h = fa.fa_read_report(report)
    exact = math.fsum(s.astype(np.float64)) + math.fsum(lo.astype(np.float64))
    got = float(h.sum_sq) + float(h.sum_sq_lo)
    assert h.nonfinite == int(c.sum())
    assert abs(got - exact) <= 1e-12 * exact


def test_merges_see_the_writes_of_the_kernel_before_them():
    """The merge kernels start early (programmatic dependent launch) and wait in the
    kernel for the grid before them.  Here that grid is a torch kernel that rewrites the
    row records right before each merge, many times over: every report must be the
    exact sum of the records just written, never of the previous ones."""
    import math
    rows = 1_048_577  # three merge levels
    rng = np.random.default_rng(31)
    rows_in = fa.stats_buffer(rows, DEV)
    scratch = fa.scratch_buffer(rows, DEV)
    report = fa.stats_buffer(1, DEV)
    base_h = (rng.random(rows) * 10).astype(np.float32)
    base = torch.from_numpy(base_h).to(DEV)
    rows_in.zero_()
    for k in range(12):
        # one elementwise kernel writes every sum, immediately before the merge
        torch.mul(base, float(k + 1), out=rows_in[:, 0].view(torch.float32))
        rows_in[k * 1000:(k + 1) * 1000, 1].fill_(k)
        fa.fa_merge_gradient_stats(rows_in, rows, scratch, report)
        h = fa.fa_read_report(report)
        # the records as written: the FP32 product, correctly rounded on both sides
        want = math.fsum((base_h * np.float32(k + 1)).astype(np.float64).tolist())
        got = float(h.sum_sq) + float(h.sum_sq_lo)
        assert abs(got - want) <= 1e-12 * want, (k, got, want)
        assert h.nonfinite == sum(range(k + 1)) * 1000


def test_statistics_capture_into_a_cuda_graph():
    """Analysis and merge captured once into a CUDA graph and replayed on new gradients
    give the same report, bit for bit, as the direct calls."""
    n = 256 * 5000 + 77
    w = CONFIG5.scaled(n, calls=3)
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    rows = fa.fa_stats_rows(n, 256)
    rb, sc, rep = fa.stats_buffer(rows, DEV), fa.scratch_buffer(rows, DEV), fa.stats_buffer(1, DEV)
    rb2, sc2, rep2 = (fa.stats_buffer(rows, DEV), fa.scratch_buffer(rows, DEV),
                      fa.stats_buffer(1, DEV))
    w.fill_grad_device(1, g)
    fa.fa_analyze_gradient(g, 256, rb)  # first use outside the capture
    fa.fa_merge_gradient_stats(rb, rows, sc, rep)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_analyze_gradient(g, 256, rb)
        fa.fa_merge_gradient_stats(rb, rows, sc, rep)
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        graph.replay()
        fa.fa_analyze_gradient(g, 256, rb2)
        fa.fa_merge_gradient_stats(rb2, rows, sc2, rep2)
        torch.cuda.synchronize()
        assert torch.equal(rep, rep2) and torch.equal(rb, rb2), call


def test_clip_decide_and_report_roundtrip(oracle_lib):
    n = 256 * 4096
    g, bits = _planted_grad(n, "bf16", 22, [], sigma=0.05)
    rows = fa.fa_stats_rows(n, 256)
    buf = fa.stats_buffer(rows, DEV)
    scratch = fa.scratch_buffer(rows, DEV)
    report = fa.stats_buffer(1, DEV)
    fa.fa_analyze_gradient(g, 256, buf)
    fa.fa_merge_gradient_stats(buf, rows, scratch, report)
    skip, norm, coef = fa.fa_clip_decide(report, 4.0, 1.0)
    s_or, c_or = oracle_lib.gradient_stats(bits, "bf16", 4.0)
    o_skip, o_norm, o_coef = oracle_lib.clip_decision(s_or, c_or, 1.0)
    assert skip == o_skip and abs(norm - o_norm) <= 1e-6 * o_norm
    assert abs(coef - o_coef) <= 1e-6 * o_coef


# ---- validation on the device -----------------------------------------------------

def _state(n):
    return [torch.randn(n, device=DEV) for _ in range(4)]


def test_rejections_leave_inputs_untouched():
    n = 4096
    p, m, v, vm = _state(n)
    g = torch.randn(n, device=DEV)
    snap = [x.clone() for x in (p, m, v, vm, g)]
    o = fa.options(amsgrad=True)
    # overlapping state buffers
    with pytest.raises(fa.FusedAdamWError) as e:
        fa.fa_adamw_step_inplace(p, g, m, m, vm, 3, o, fa.control())
    assert e.value.status == 5
    big = torch.randn(2 * n, device=DEV)
    with pytest.raises(fa.FusedAdamWError) as e:
        fa.fa_adamw_step_inplace(big[:n], g, big[n // 2:n // 2 + n], v, vm, 3, o, fa.control())
    assert e.value.status == 5
    # gradient aliasing the parameters
    with pytest.raises(fa.FusedAdamWError) as e:
        fa.fa_adamw_step_inplace(p, p, m, v, vm, 3, o, fa.control())
    assert e.value.status == 5
    # host memory (pageable and pinned)
    for host in (torch.randn(n), torch.randn(n).pin_memory()):
        with pytest.raises((fa.FusedAdamWError, ValueError)):
            fa.fa_adamw_step_inplace(p, host, m, v, vm, 3, o, fa.control())
    # out of place: output aliasing an input
    with pytest.raises(fa.FusedAdamWError) as e:
        import ctypes
        from amsgrad_optimizer_step_gb300 import _lib
        tt, up = ctypes.c_uint64(), ctypes.c_int32()
        st = _lib.load().fa_adamw_step(n, p.data_ptr(), g.data_ptr(), 0, m.data_ptr(),
                                       v.data_ptr(), vm.data_ptr(), 3, ctypes.byref(o),
                                       fa.control(), p.data_ptr(), m.data_ptr(),
                                       v.data_ptr(), vm.data_ptr(), ctypes.byref(tt),
                                       ctypes.byref(up), None)
        _lib.check("fa_adamw_step", st)
    assert e.value.status == 5
    # misaligned FP32 pointer (2-byte offset)
    import ctypes
    from amsgrad_optimizer_step_gb300 import _lib
    tt = ctypes.c_uint64(3)
    up = ctypes.c_int32()
    st = _lib.load().fa_adamw_step_inplace(n - 1, p.data_ptr() + 2, g.data_ptr(), 0, m.data_ptr(),
                                           v.data_ptr(), vm.data_ptr(), ctypes.byref(tt),
                                           ctypes.byref(o), fa.control(), 1.0, ctypes.byref(up),
                                           None)
    assert st == 7 and tt.value == 3
    torch.cuda.synchronize()
    for a, b in zip((p, m, v, vm, g), snap):
        assert torch.equal(a, b)


def test_analyze_rejects_plan_overflow():
    n = 4_194_305 * 2
    g = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    buf = fa.stats_buffer(1, DEV)
    with pytest.raises(fa.FusedAdamWError) as e:
        fa.fa_analyze_gradient(g, 2, buf)
    assert e.value.status == 8


def test_host_pointers_rejected_by_the_library():
    """The C ABI itself refuses host memory (pageable or pinned) with FA_ERR_POINTER."""
    import ctypes
    from amsgrad_optimizer_step_gb300 import _lib
    n = 1024
    p, m, v, _ = _state(n)
    o = fa.options()
    for host in (torch.randn(n), torch.randn(n).pin_memory()):
        tt = ctypes.c_uint64(2)
        up = ctypes.c_int32(5)
        st = _lib.load().fa_adamw_step_inplace(n, p.data_ptr(), host.data_ptr(), 0, m.data_ptr(),
                                               v.data_ptr(), None, ctypes.byref(tt),
                                               ctypes.byref(o), fa.control(), 1.0,
                                               ctypes.byref(up), None)
        assert st == 6 and tt.value == 2 and up.value == 5


# ---- fused low-precision write-back ------------------------------------------------

@pytest.mark.parametrize("model_dtype", ["bf16", "f16"])
def test_writeback_scaled_flat(model_dtype):
    w = dataclasses.replace(CONFIG3, calls=6)
    s = run_workload(w, 1_000_003, "bucket", DEV, guard=1024, model_dtype=model_dtype)
    assert s["t"] == 6


def test_writeback_scaled_decoder_bucket_with_skip():
    off = small_decoder_offsets()
    w = dataclasses.replace(CONFIG4_MAX, skip_calls=(3,), calls=5)
    s = run_workload(w, int(off[-1]), "bucket", DEV, segments=off, guard=1024,
                     model_dtype="f16")
    assert s["t"] == 4 and s["skips"] == 1


def test_writeback_full_size_sampled():
    idx = sample_indices(CONFIG4.n, seed=6)
    w = dataclasses.replace(CONFIG4, calls=3)
    s = run_workload(w, w.n, "bucket", DEV, idx=idx, model_dtype="bf16")
    assert s["t"] == 3


@pytest.mark.parametrize("n", [1, 7, 9, 4097])
@pytest.mark.parametrize("model_dtype", ["bf16", "f16"])
def test_writeback_edge_sizes(n, model_dtype):
    w = dataclasses.replace(CONFIG1, grad_dtype="bf16", calls=3, inplace=True)
    run_workload(w, n, "bucket", DEV, guard=64, model_dtype=model_dtype)


def test_writeback_misaligned_model_view(oracle_lib):
    """A model copy starting 2 bytes off a 16-byte boundary takes the scalar kernel."""
    n = 20_001
    w = dataclasses.replace(CONFIG3, calls=2).scaled(n)
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p)
    m, v = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    full = torch.zeros(n + 8, dtype=torch.bfloat16, device=DEV)
    model = full[1:1 + n]
    t = 0
    for call in (1, 2):
        w.fill_grad_device(call, g)
        assert fa.fa_bucket_update(None, p, g, m, v, None, t, fa.options(**w.options()),
                                   fa.control(), p_model=model)
        t += 1
    torch.cuda.synchronize()
    bits = model.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(bits, oracle_lib.model_copy(p.cpu().numpy(), "bf16"))


def test_writeback_rejections():
    n = 1024
    p, m, v, _ = _state(n)
    g = torch.randn(n, device=DEV)
    model = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    o = fa.options()
    import ctypes
    from amsgrad_optimizer_step_gb300 import _lib
    up = ctypes.c_int32()
    u = _lib.FaBucketUpdate(n_total=n, p=p.data_ptr(), g=g.data_ptr(), gdt=0, m=m.data_ptr(),
                            v=v.data_ptr(), t=1, grad_mult=1.0, p_model=model.data_ptr(),
                            model_dtype=0)
    st = _lib.load().fa_bucket_update(ctypes.byref(u), ctypes.byref(o), fa.control(),
                                      ctypes.byref(up), None)
    assert st == 2  # FP32 is not a model-copy dtype
    with pytest.raises(fa.FusedAdamWError) as e:
        fa.fa_bucket_update(None, p, g, m, v, None, 1, o, fa.control(),
                            p_model=p.view(torch.bfloat16)[:n])
    assert e.value.status == 5
    assert not model.view(torch.int16).any()


# ---- staged comparison ---------------------------------------------------------------

@pytest.mark.parametrize("gdt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("ams", [False, True])
def test_staged_equals_fused_bitwise(gdt, ams):
    """The 4/5-kernel staged baseline evaluates the fused kernel's FP32 operations
    stage by stage: same results bit for bit, first step included."""
    w, p0 = _fresh(70_001, gdt, 17, ams=ams)
    o = fa.options(**dict(w.options(), maximize=True))
    pa, pb = p0.clone(), p0.clone()
    sa, sb = _zeros(w.n, 3), _zeros(w.n, 3)
    if not ams:
        sa[2] = sb[2] = None
    delta = torch.empty(w.n, device=DEV)
    ta = tb = 0
    for call in range(1, 5):
        g = _grads(w, call)
        ta, _ = fa.fa_adamw_step_inplace(pa, g, *sa, ta, o, fa.control(2.0), grad_mult=0.75)
        tb, _ = fa.fa_adamw_step_staged(pb, g, *sb, tb, o, fa.control(2.0), delta, grad_mult=0.75)
    torch.cuda.synchronize()
    assert ta == tb == 4
    assert torch.equal(pa.view(torch.int32), pb.view(torch.int32))
    for x, y in zip(sa, sb):
        if x is not None:
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("n", [70_001, 1_000_003])
@pytest.mark.parametrize("ams", [False, True])
@pytest.mark.parametrize("gdt", ["f32", "f16", "bf16"])
def test_staged_vs_oracle(gdt, ams, n):
    """The staged 4/5-kernel comparison against the oracle itself, not only against
    the fused kernel: every element of every call, one step from identical state
    (1e-6 and the FP32 error bound) and along the oracle's own trajectory (1e-5).
    Lengths leave a scalar tail after the 4-element vectors; gradients stored x128
    with gradient_scale 128, a clip factor of 0.75, a skipped third call, and
    maximize on the FP16 runs."""
    w = dataclasses.replace(CONFIG2, name=f"staged_{gdt}", grad_dtype=gdt, amsgrad=ams, calls=5,
                            skip_calls=(3,), maximize=gdt == "f16")
    s = run_workload(w, n, "staged", DEV, guard=1024, grad_mult=0.75)
    assert s["updates"] == 4 and s["skips"] == 1 and s["t"] == 4


def test_staged_rejects_unaligned_views():
    n = 4096
    full = torch.zeros(n + 4, device=DEV)
    p = full[1:1 + n]
    m, v = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    g = torch.zeros(n, device=DEV)
    delta = torch.empty(n, device=DEV)
    with pytest.raises(fa.FusedAdamWError) as e:
        fa.fa_adamw_step_staged(p, g, m, v, None, 0, fa.options(), fa.control(), delta)
    assert e.value.status == 7


def test_update_pipeline_never_gave_up():
    """After everything above, no bounded wait in the shared-memory pipeline gave up."""
    assert fa.fa_device_error() == 0


# ---- device-gated update ---------------------------------------------------------------

@pytest.mark.parametrize("max_norm", [1.0, 0.0, 1e6])
def test_gated_step_equals_host_decided_step_bitwise(max_norm):
    """Same report, same FP64 decision on the device: bit-identical to reading the
    report back first, including the skipped call with a planted +Inf."""
    n = 256 * 5000 + 77
    w = CONFIG5.scaled(n, calls=4, inf_call=2)
    dev_state = []
    mailbox = fa.report_mailbox()
    for gated in (False, True):
        p = torch.empty(n, device=DEV)
        w.fill_params_device(p)
        m, v = torch.empty_like(p), torch.empty_like(p)
        g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        rows = fa.fa_stats_rows(n, 256)
        rb, sc, rep = fa.stats_buffer(rows, DEV), fa.scratch_buffer(rows, DEV), fa.stats_buffer(1, DEV)
        t = 0
        reports = []
        for call in range(1, w.calls + 1):
            w.fill_grad_device(call, g)
            fn = (lambda *a: fa.fa_bucket_step_clipped_gated(*a, mailbox)) if gated \
                else fa.fa_bucket_step_clipped
            t, r = fn(None, p, g, m, v, None, t, fa.options(**w.options()), fa.control(),
                      max_norm, 256, rb, sc, rep)
            reports.append((r.updated, r.skipped_nonfinite, r.nonfinite, repr(r.grad_norm),
                            repr(r.clip_coef)))  # repr: a skipped step's norm is NaN
        torch.cuda.synchronize()
        dev_state.append((t, reports, p.clone(), m.clone(), v.clone()))
    (ta, ra, *sa), (tb, rb_, *sb) = dev_state
    assert ta == tb == 3 and ra == rb_
    assert ra[1][1] == 1  # the +Inf call was skipped
    for x, y in zip(sa, sb):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("scale", [2.0 ** -3, 128.0, 2.0 ** 40, 3.0, 1000.0, 0.1])
@pytest.mark.parametrize("amsgrad", [False, True])
def test_gated_step_equals_host_decided_step_bitwise_at_any_scale(scale, amsgrad):
    """The device takes the decision's divisions by the gradient scale as multiplications
    by the exact inverse when the scale is a power of two (and then runs the full grid),
    and as divisions otherwise (the TMA pipeline and persistent CTAs).  Either way the
    steps are bit-identical to the host's decision, first step, clipped steady steps and
    the skipped +Inf call alike."""
    n = 256 * 5000 + 77  # more than two tiles per SM: the steady steps reach the pipeline
    w = dataclasses.replace(CONFIG5, gradient_scale=scale, grad_premul=scale,
                            amsgrad=amsgrad).scaled(n, calls=4, inf_call=2)
    o = fa.options(**w.options())
    mailbox = fa.report_mailbox()
    states = []
    for gated in (False, True):
        p = torch.empty(n, device=DEV)
        w.fill_params_device(p)
        m, v = torch.empty_like(p), torch.empty_like(p)
        vmax = torch.empty_like(p) if amsgrad else None
        g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        rows = fa.fa_stats_rows(n, 256)
        rb, sc, rep = fa.stats_buffer(rows, DEV), fa.scratch_buffer(rows, DEV), fa.stats_buffer(1, DEV)
        t, reports = 0, []
        for call in range(1, w.calls + 1):
            w.fill_grad_device(call, g)
            fn = (lambda *a: fa.fa_bucket_step_clipped_gated(*a, mailbox)) if gated \
                else fa.fa_bucket_step_clipped
            t, r = fn(None, p, g, m, v, vmax, t, o, fa.control(scale), 0.05, 256, rb, sc, rep)
            reports.append((r.updated, r.skipped_nonfinite, repr(r.grad_norm), repr(r.clip_coef)))
        torch.cuda.synchronize()
        states.append((t, reports, [x.clone() for x in (p, m, v, vmax) if x is not None]))
    (ta, ra, sa), (tb, rb_, sb) = states
    assert ta == tb == 3 and ra == rb_
    assert ra[1][1] == 1 and all(0 < float(c) < 1 for _, s_, _, c in ra if not s_), ra
    for x, y in zip(sa, sb):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("off", [0, 1, 3])
@pytest.mark.parametrize("n", [1023, 1025, 2049, 3 * 1024 + 5])
def test_full_grid_stretch_edges_and_scalar_heads(n, off, oracle_lib):
    """The full grid gives each 64-thread CTA 1024 elements.  Sizes on both sides of one,
    two and three stretches, with p, m and v viewed ``off`` elements past a 16-byte
    boundary and the BF16 gradient at the offset that keeps all four co-aligned, so that
    a scalar head of (4 - off) % 4 elements comes before the vector body; the elements
    around the views are guards.  Decided on the host and on the device (four calls, a
    +Inf in the third, the clip active): the two bit-identical, and both on the oracle's
    trajectory."""
    import oracle
    from gpu_harness import gate
    goff = off + 4 if off % 4 else 0  # 2-byte elements: the same 16-byte phase as p's
    w = CONFIG5.scaled(n, calls=4, inf_call=3)
    w = dataclasses.replace(w, max_grad_norm=0.02)  # the clip is active at these sizes
    opts = w.options()
    idx = np.arange(n)
    rows = fa.fa_stats_rows(n, 256)
    states = []
    mailbox = fa.report_mailbox()
    for gated in (False, True):
        full = [torch.full((n + 32,), -7.0, device=DEV) for _ in range(3)]
        p, m, v = (x[off:off + n] for x in full)
        w.fill_params_device(p)
        gfull = torch.zeros(n + 32, dtype=torch.bfloat16, device=DEV)
        g = gfull[goff:goff + n]
        rb, sc, rep = fa.stats_buffer(rows, DEV), fa.scratch_buffer(rows, DEV), fa.stats_buffer(1, DEV)
        ref = oracle.OracleAdamW(w.params_host(idx), opts, lib_=oracle_lib)
        t = 0
        for call in range(1, w.calls + 1):
            w.fill_grad_device(call, g)
            step = (lambda *a: fa.fa_bucket_step_clipped_gated(*a, mailbox)) if gated \
                else fa.fa_bucket_step_clipped
            t, r = step(None, p, g, m, v, None, t, fa.options(**opts), fa.control(),
                        w.max_grad_norm, 256, rb, sc, rep)
            gh = w.grad_host(call, idx)
            st, c = oracle_lib.gradient_stats(gh, "bf16", 1.0)
            skip, _, coef = oracle_lib.clip_decision(st, c, w.max_grad_norm)
            assert bool(r.skipped_nonfinite) == skip == (call == 3)
            ref.step(gh, "bf16", skip_update=skip, clip_coef=coef)
        torch.cuda.synchronize()
        assert t == ref.state.t == 3
        for x in full:  # the elements around the view are untouched
            assert torch.all(x[:off] == -7.0) and torch.all(x[off + n:] == -7.0)
        gate(p.cpu().numpy(), ref.p, 1e-5, f"n={n} off={off} gated={gated} p")
        gate(m.cpu().numpy(), ref.state.m, 1e-5, "m")
        gate(v.cpu().numpy(), ref.state.v, 1e-5, "v")
        states.append([x.clone() for x in (p, m, v)])
    for a, b in zip(*states):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_gated_step_full_size_bitwise():
    """The benchmark's launch configuration: the 1,073,741,824-parameter workload, rows of
    256, the update gated on the device report, five calls with the +Inf in call 3;
    bit-identical at every call to the host-decided step (itself checked against the
    oracle at this size in test_config5_full_size_sampled)."""
    w = CONFIG5
    n = w.n
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    states = []
    for _ in range(2):
        p = torch.empty(n, device=DEV)
        w.fill_params_device(p)
        rows = fa.fa_stats_rows(n, w.row_len)
        states.append({"p": p, "m": torch.empty_like(p), "v": torch.empty_like(p), "t": 0,
                       "rows": fa.stats_buffer(rows, DEV), "scr": fa.scratch_buffer(rows, DEV),
                       "rep": fa.stats_buffer(1, DEV)})
    o = fa.options(**w.options())
    mailbox = fa.report_mailbox()
    gated = lambda *a: fa.fa_bucket_step_clipped_gated(*a, mailbox)  # noqa: E731
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        reps = []
        for s_, fn in zip(states, (fa.fa_bucket_step_clipped, gated)):
            s_["t"], r = fn(None, s_["p"], g, s_["m"], s_["v"], None, s_["t"], o, fa.control(),
                            w.max_grad_norm, w.row_len, s_["rows"], s_["scr"], s_["rep"])
            reps.append((r.updated, r.skipped_nonfinite, r.nonfinite, repr(r.grad_norm),
                         repr(r.clip_coef)))
        torch.cuda.synchronize()
        assert reps[0] == reps[1], (call, reps)
        assert reps[0][1] == (call == w.inf_call)
        a, b = states
        assert a["t"] == b["t"]
        for k in ("p", "m", "v"):
            assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), (call, k)
    assert states[0]["t"] == 4


@pytest.mark.parametrize("model_dtype", [torch.bfloat16, torch.float16])
def test_gated_writeback_equals_host_decided_writeback_bitwise(model_dtype):
    """The model-copy update gated on the device report: parameters, moments and the
    low-precision copy bit-identical to deciding on the host, the +Inf call included."""
    n = 256 * 4000 + 33
    w = CONFIG5.scaled(n, calls=4, inf_call=2)
    states = []
    for gated in (False, True):
        p = torch.empty(n, device=DEV)
        w.fill_params_device(p)
        m, v = torch.empty_like(p), torch.empty_like(p)
        model = torch.zeros(n, dtype=model_dtype, device=DEV)
        g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        rows = fa.fa_stats_rows(n, 256)
        rb, sc, rep = (fa.stats_buffer(rows, DEV), fa.scratch_buffer(rows, DEV),
                       fa.stats_buffer(1, DEV))
        t = 0
        for call in range(1, w.calls + 1):
            w.fill_grad_device(call, g)
            fa.fa_analyze_gradient(g, 256, rb)
            fa.fa_merge_gradient_stats(rb, rows, sc, rep)
            o = fa.options(**w.options())
            if gated:
                fa.fa_bucket_update(None, p, g, m, v, None, t, o, fa.control(), report=rep,
                                    max_grad_norm=0.5, p_model=model)
                h = fa.fa_read_report(rep)
                skip, _, _ = fa.fa_clip_decision(fa.fa_stats_sum_sq(h), h.nonfinite, 1.0, 0.5)
                t += 0 if skip else 1
            else:
                skip, _, coef = fa.fa_clip_decide(rep, 1.0, 0.5)
                if not skip:
                    assert fa.fa_bucket_update(None, p, g, m, v, None, t, o, fa.control(),
                                               grad_mult=coef, p_model=model)
                    t += 1
        torch.cuda.synchronize()
        states.append((t, p.clone(), m.clone(), v.clone(), model.clone()))
    (ta, *a), (tb, *b) = states
    assert ta == tb == 3
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.element_size() == 2 else x.view(torch.int32),
                           y.view(torch.int16) if y.element_size() == 2 else y.view(torch.int32))


def test_gated_update_skips_on_non_finite_report():
    n = 4_000_000
    p = torch.randn(n, device=DEV)
    m, v = torch.randn(n, device=DEV), torch.rand(n, device=DEV)
    g = torch.randn(n, device=DEV).to(torch.bfloat16)
    snap = [x.clone() for x in (p, m, v)]
    report = torch.zeros((1, 3), dtype=torch.int32, device=DEV)
    report[0, 1] = 2  # two non-finite values
    fa.fa_bucket_update(None, p, g, m, v, None, 4, fa.options(), fa.control(), report=report,
                        max_grad_norm=1.0)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip((p, m, v), snap))
    report[0, 1] = 0
    report[0, 0] = torch.tensor([4.0], dtype=torch.float32).view(torch.int32)
    fa.fa_bucket_update(None, p, g, m, v, None, 4, fa.options(), fa.control(), report=report,
                        max_grad_norm=1.0)
    torch.cuda.synchronize()
    assert not torch.equal(p, snap[0])


def test_report_mailbox_rules():
    """The one-call device-gated step reads its report through the caller's mailbox:
    pageable host memory, device memory and NULL are rejected before anything is
    enqueued (state untouched); a sequence word at 2^32 - 1 wraps to 0; calls in a row
    on one mailbox each read their own report."""
    import ctypes
    from amsgrad_optimizer_step_gb300 import _lib
    n = 256 * 4000 + 5
    w = CONFIG5.scaled(n, calls=3, inf_call=2)
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p)
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    w.fill_grad_device(1, g)
    rows = fa.fa_stats_rows(n, 256)
    rb, sc, rep = fa.stats_buffer(rows, DEV), fa.scratch_buffer(rows, DEV), fa.stats_buffer(1, DEV)
    o = fa.options(**w.options())
    lib = _lib.load()
    snap = [x.clone() for x in (p, m, v)]

    def raw(mailbox_ptr):
        tt = ctypes.c_uint64(0)
        out = fa.FaStepReport()
        return lib.fa_bucket_step_clipped_gated(
            None, 0, n, p.data_ptr(), g.data_ptr(), 2, m.data_ptr(), v.data_ptr(), None,
            ctypes.byref(tt), ctypes.byref(o), fa.control(), w.max_grad_norm, 256,
            rb.data_ptr(), rb.shape[0], sc.data_ptr(), sc.numel(), rep.data_ptr(),
            mailbox_ptr, ctypes.byref(out), None)

    pageable = np.zeros(4, np.uint32)
    assert raw(pageable.ctypes.data) == 6            # FA_ERR_POINTER: not pinned
    assert raw(torch.zeros(4, dtype=torch.int32, device=DEV).data_ptr()) == 6  # device memory
    assert raw(None) == 1                             # FA_ERR_NULL
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip((p, m, v), snap))
    with pytest.raises(ValueError):
        fa.fa_bucket_step_clipped_gated(None, p, g, m, v, None, 0, o, fa.control(),
                                        w.max_grad_norm, 256, rb, sc, rep,
                                        torch.zeros(4, dtype=torch.int32))  # not pinned

    mailbox = fa.report_mailbox()
    mailbox[3] = -1  # sequence word 2^32 - 1: the next post is 0
    t = 0
    reports = []
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        t, r = fa.fa_bucket_step_clipped_gated(None, p, g, m, v, None, t, o, fa.control(),
                                               w.max_grad_norm, 256, rb, sc, rep, mailbox)
        reports.append((r.skipped_nonfinite, r.nonfinite, r.grad_norm))
        assert int(mailbox[3]) == call - 1  # 0, 1, 2
    torch.cuda.synchronize()
    assert t == 2 and [x[0] for x in reports] == [0, 1, 0] and reports[1][1] == 1
    assert reports[0][2] > 0 and reports[2][2] > 0 and reports[0][2] != reports[2][2]
