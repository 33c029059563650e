"""The torch.optim-style FusedAdamW and its GradScaler, against the oracle."""

import io

import numpy as np
import pytest
import torch

import oracle
from amsgrad_optimizer_step_gb300.optim import FusedAdamW, GradScaler
from gpu_harness import gate

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
SHAPES = [(33, 17), (129,), (8, 1000), (5,), (64, 64)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from amsgrad_optimizer_step_gb300 import build
    build.build()


def _params(seed, dtype=torch.float32, shapes=SHAPES):
    g = torch.Generator().manual_seed(seed)
    return [torch.nn.Parameter((torch.randn(s, generator=g) * 0.02).to(dtype).to(DEV))
            for s in shapes]


def _grads(seed, step, shapes=SHAPES, scale=1.0):
    g = torch.Generator().manual_seed(1000 * seed + step)
    return [(torch.randn(s, generator=g) * 1e-2 * scale).to(torch.float32) for s in shapes]


def _set_grads(params, grads):
    for p, gr in zip(params, grads):
        p.grad.copy_(gr.to(p.dtype).to(DEV))


def _host(t):
    return t.detach().float().cpu().numpy().reshape(-1)


@pytest.mark.parametrize("amsgrad,maximize", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("clip", [None, 0.05])
def test_matches_oracle_per_parameter(amsgrad, maximize, clip):
    params = _params(1)
    hp = dict(lr=2e-3, betas=(0.9, 0.99), eps=1e-6, weight_decay=0.01, amsgrad=amsgrad,
              maximize=maximize)
    opt = FusedAdamW(params, max_grad_norm=clip, **hp)
    lib = oracle.lib()
    oo = dict(lr=2e-3, beta1=0.9, beta2=0.99, eps=1e-6, weight_decay=0.01, amsgrad=amsgrad,
              maximize=maximize)
    refs = [oracle.OracleAdamW(_host(p), oo, lib_=lib) for p in params]
    for step in range(1, 7):
        grads = _grads(1, step)
        _set_grads(params, grads)
        opt.step()
        coef = 1.0
        if clip is not None:
            allg = np.concatenate([g.numpy().reshape(-1) for g in grads])
            s, c = lib.gradient_stats(allg, "f32")
            _, norm, coef = lib.clip_decision(s, c, clip)
            assert abs(opt.last_report["grad_norm"] - norm) <= 1e-5 * norm
            assert coef < 1.0
        for r, g in zip(refs, grads):
            r.step(g.numpy().reshape(-1), "f32", clip_coef=coef)
        torch.cuda.synchronize()
        for p, r in zip(params, refs):
            gate(_host(p), r.p, 1e-5, f"p step {step}")
            st = opt.state[p]
            gate(_host(st["exp_avg"]), r.state.m, 1e-5, "m")
            gate(_host(st["exp_avg_sq"]), r.state.v, 1e-5, "v")
            if amsgrad:
                gate(_host(st["max_exp_avg_sq"]), r.state.vmax, 1e-5, "vmax")
    assert float(opt.state_dict()["state"][0]["step"]) == 6


def test_real_autograd_accumulates_into_the_bucket():
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(40, 64), torch.nn.Tanh(),
                                torch.nn.Linear(64, 3)).to(DEV)
    opt = FusedAdamW(model.parameters(), lr=1e-2, max_grad_norm=1.0)
    bucket = opt._buckets[0]
    lo, hi = bucket.grad.data_ptr(), bucket.grad.data_ptr() + bucket.grad.numel() * 4
    x = torch.randn(16, 40, device=DEV)
    y = torch.randn(16, 3, device=DEV)
    losses = []
    for _ in range(30):
        opt.zero_grad()
        loss = torch.nn.functional.mse_loss(model(x), y)
        loss.backward()
        for p in model.parameters():
            assert lo <= p.grad.data_ptr() < hi, "gradient left the bucket"
        opt.step()
        losses.append(float(loss.detach()))
    assert losses[-1] < 0.5 * losses[0]
    assert opt.last_report["skipped"] is False and opt.last_report["grad_norm"] is not None


def test_param_groups_share_one_global_clip():
    a = _params(2, shapes=[(100,), (7, 9)])
    b = _params(3, shapes=[(300,)])
    opt = FusedAdamW([{"params": a, "lr": 1e-3}, {"params": b, "lr": 5e-3, "weight_decay": 0.1}],
                     max_grad_norm=0.01)
    lib = oracle.lib()
    ga = _grads(2, 1, shapes=[(100,), (7, 9)])
    gb = _grads(3, 1, shapes=[(300,)])
    ra = [oracle.OracleAdamW(_host(p), dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-5,
                                            weight_decay=1e-4, amsgrad=False, maximize=False),
                             lib_=lib) for p in a]
    rb = [oracle.OracleAdamW(_host(p), dict(lr=5e-3, beta1=0.9, beta2=0.999, eps=1e-5,
                                            weight_decay=0.1, amsgrad=False, maximize=False),
                             lib_=lib) for p in b]
    _set_grads(a, ga)
    _set_grads(b, gb)
    opt.step()
    allg = np.concatenate([g.numpy().reshape(-1) for g in ga + gb])
    s, c = lib.gradient_stats(allg, "f32")
    _, norm, coef = lib.clip_decision(s, c, 0.01)
    for r, g, p in zip(ra + rb, ga + gb, a + b):
        r.step(g.numpy().reshape(-1), "f32", clip_coef=coef)
        gate(_host(p), r.p, 1e-6, "grouped p")


def test_grad_scaler_skips_non_finite_and_backs_off():
    params = _params(4)
    opt = FusedAdamW(params, lr=1e-3)
    scaler = GradScaler(init_scale=1024.0, growth_interval=2)
    lib = oracle.lib()
    oo = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=1e-4, amsgrad=False,
              maximize=False)
    refs = [oracle.OracleAdamW(_host(p), oo, lib_=lib) for p in params]
    scales = []
    for step in range(1, 7):
        s = scaler.get_scale()
        grads = _grads(4, step, scale=s)
        if step == 3:
            grads[2][1, 5] = float("inf")
        before = [p.detach().clone() for p in params]
        _set_grads(params, grads)
        scaler.step(opt)
        skipped = opt.last_report["skipped"]
        assert skipped == (step == 3)
        for r, g in zip(refs, grads):
            r.step(g.numpy().reshape(-1), "f32", gradient_scale=s, skip_update=skipped)
        torch.cuda.synchronize()
        if skipped:
            assert all(torch.equal(p, q) for p, q in zip(params, before))
            assert opt.last_report["nonfinite"] == 1
        for p, r in zip(params, refs):
            gate(_host(p), r.p, 1e-5, f"scaled p step {step}")
        scaler.update()
        scales.append(scaler.get_scale())
    assert scales[:3] == [1024.0, 2048.0, 1024.0]


def _train(opt, params, steps, first=1):
    for step in range(first, first + steps):
        _set_grads(params, _grads(5, step))
        opt.step()
    torch.cuda.synchronize()


def test_state_dict_round_trip_bitwise():
    ref_params = _params(5)
    ref = FusedAdamW(ref_params, amsgrad=True, max_grad_norm=0.5, hierarchical_stats=True)
    _train(ref, ref_params, 10)

    params = _params(5)
    opt = FusedAdamW(params, amsgrad=True, max_grad_norm=0.5, hierarchical_stats=True)
    _train(opt, params, 5)
    buf = io.BytesIO()
    torch.save({"model": [p.detach().cpu() for p in params], "opt": opt.state_dict()}, buf)
    sd = opt.state_dict()
    assert sd["fused_options"]["step_options_version"] == 2
    buf.seek(0)
    saved = torch.load(buf, weights_only=False)
    fresh = _params(99)  # different initial values, overwritten by the checkpoint
    with torch.no_grad():
        for p, q in zip(fresh, saved["model"]):
            p.copy_(q)
    opt2 = FusedAdamW(fresh, amsgrad=True)
    opt2.load_state_dict(saved["opt"])
    assert opt2.max_grad_norm == 0.5 and opt2.hierarchical_stats
    _train(opt2, fresh, 5, first=6)
    for p, q in zip(fresh, ref_params):
        assert torch.equal(p, q)
    for p, q in zip(fresh, ref_params):
        assert torch.equal(opt2.state[p]["exp_avg_sq"], ref.state[q]["exp_avg_sq"])


def test_old_state_dict_turns_fused_modes_off():
    params = _params(6)
    opt = FusedAdamW(params, max_grad_norm=1.0, hierarchical_stats=True)
    _train(opt, params, 2)
    sd = opt.state_dict()
    del sd["fused_options"]
    opt2 = FusedAdamW(_params(6), max_grad_norm=1.0, hierarchical_stats=True)
    opt2.load_state_dict(sd)
    assert opt2.max_grad_norm is None and opt2.hierarchical_stats is False
    sd1 = opt.state_dict()
    sd1["fused_options"]["step_options_version"] = 1
    opt3 = FusedAdamW(_params(6))
    opt3.load_state_dict(sd1)
    assert opt3.hierarchical_stats is False and opt3.max_grad_norm == 1.0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_low_precision_params_keep_fp32_masters(dtype):
    params = _params(7, dtype=dtype)
    masters0 = [_host(p) for p in params]
    opt = FusedAdamW(params, lr=1e-3)
    lib = oracle.lib()
    oo = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=1e-4, amsgrad=False,
              maximize=False)
    refs = [oracle.OracleAdamW(m, oo, lib_=lib) for m in masters0]
    name = "bf16" if dtype == torch.bfloat16 else "f16"
    for step in range(1, 5):
        grads = [g.to(dtype) for g in _grads(7, step)]
        _set_grads(params, grads)
        opt.step()
        for r, g in zip(refs, grads):
            bits = g.view(torch.int16).numpy().view(np.uint16).reshape(-1)
            r.step(bits, name)
    torch.cuda.synchronize()
    for p, r in zip(params, refs):
        master = opt.state[p]["master_param"]
        gate(_host(master), r.p, 1e-5, "master")
        bits = p.detach().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
        assert np.array_equal(bits, lib.model_copy(_host(master), name))


def test_empty_and_gradless_parameters():
    """A zero-element parameter and one that never receives a gradient share a bucket
    with ordinary ones: the empty one is carried along untouched, the gradless one is
    inactive (not updated, its step count stays 0, it adds nothing to the global norm),
    the rest are updated as usual."""
    shapes = [(0,), (17,), (3, 5)]
    params = _params(13, shapes=shapes)
    before = params[2].detach().clone()
    opt = FusedAdamW(params, lr=1e-2, weight_decay=0.1, max_grad_norm=1.0)
    lib = oracle.lib()
    oo = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=0.1, amsgrad=False,
              maximize=False)
    ref = oracle.OracleAdamW(_host(params[1]), oo, lib_=lib)
    for step in range(1, 4):
        g17 = (torch.randn(17, generator=torch.Generator().manual_seed(step)) * 1e-2)
        params[0].grad = None
        params[1].grad = g17.to(DEV)        # a new tensor: gathered into the bucket
        params[2].grad = None               # never receives a gradient
        opt.step()
        s, c = lib.gradient_stats(g17.numpy(), "f32")
        _, norm, coef = lib.clip_decision(s, c, 1.0)
        assert abs(opt.last_report["grad_norm"] - norm) <= 1e-5 * norm
        ref.step(g17.numpy(), "f32", clip_coef=coef)
    torch.cuda.synchronize()
    assert params[0].numel() == 0
    gate(_host(params[1]), ref.p, 1e-5, "p")
    assert torch.equal(params[2], before)
    assert not opt.state[params[2]]["exp_avg"].any()
    steps = [float(st["step"]) for st in opt.state_dict()["state"].values()]
    assert steps[1:] == [3.0, 0.0]


ACTIVITY = [  # which of the five parameters have a gradient, step by step
    [True, True, True, True, True],
    [True, False, True, False, True],
    [False, True, True, True, False],
    [True, True, True, True, True],
    [True, True, False, True, True],
]


@pytest.mark.parametrize("dtype,clip", [(torch.float32, None), (torch.float32, 0.05),
                                        (torch.bfloat16, 0.05)])
def test_intermittent_parameters_keep_their_own_step_counts(dtype, clip):
    """Parameters that miss some steps are updated with their own step counts (their
    own bias corrections), by one launch per run of active parameters with equal
    counts; the global norm covers only the active parameters of each step."""
    params = _params(15, dtype=dtype)
    hp = dict(lr=2e-3, betas=(0.9, 0.99), eps=1e-6, weight_decay=0.01, amsgrad=True)
    opt = FusedAdamW(params, max_grad_norm=clip, **hp)
    lib = oracle.lib()
    oo = dict(lr=2e-3, beta1=0.9, beta2=0.99, eps=1e-6, weight_decay=0.01, amsgrad=True,
              maximize=False)
    name = "f32" if dtype == torch.float32 else "bf16"
    refs = [oracle.OracleAdamW(_host(p), oo, lib_=lib) for p in params]
    for step, act in enumerate(ACTIVITY, start=1):
        grads = _grads(15, step)
        opt.zero_grad(set_to_none=True)
        bits = []
        for p, g, a in zip(params, grads, act):
            if a:
                p.grad = g.to(dtype).to(DEV)
                bits.append(lib_bits(p.grad, name))
        opt.step()
        coef = 1.0
        if clip is not None:
            s, c = lib.gradient_stats(np.concatenate(bits), name)
            _, norm, coef = lib.clip_decision(s, c, clip)
            assert abs(opt.last_report["grad_norm"] - norm) <= 1e-5 * norm
        k = 0
        for r, a in zip(refs, act):
            if a:
                r.step(bits[k], name, clip_coef=coef)
                k += 1
    torch.cuda.synchronize()
    for p, r in zip(params, refs):
        st = opt.state[p]
        master = st["master_param"] if dtype != torch.float32 else p
        gate(_host(master), r.p, 1e-5, "p")
        gate(_host(st["exp_avg"]), r.state.m, 1e-5, "m")
        gate(_host(st["max_exp_avg_sq"]), r.state.vmax, 1e-5, "vmax")
        if dtype != torch.float32:
            got = p.detach().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
            assert np.array_equal(got, lib.model_copy(_host(master), name))
    want = [sum(a[i] for a in ACTIVITY) for i in range(5)]
    assert [int(float(st["step"])) for st in opt.state_dict()["state"].values()] == want
    assert want == [r.state.t for r in refs]


def _train_intermittent(opt, params, steps, first=1, dtype=torch.float32):
    for step in range(first, first + steps):
        act = ACTIVITY[(step - 1) % len(ACTIVITY)]
        opt.zero_grad(set_to_none=True)
        for p, g, a in zip(params, _grads(16, step), act):
            if a:
                p.grad = g.to(dtype).to(DEV)
        opt.step()
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_state_dict_round_trip_with_different_step_counts(dtype):
    """Parameters with different step counts survive save / load: 3 intermittent steps
    (counts 2 and 3), a checkpoint into a fresh optimizer, 7 more, bit-identical to 10
    uninterrupted."""
    hp = dict(lr=1e-3, amsgrad=True, max_grad_norm=0.5)
    ref_params = _params(16, dtype=dtype)
    ref = FusedAdamW(ref_params, **hp)
    _train_intermittent(ref, ref_params, 10, dtype=dtype)

    params = _params(16, dtype=dtype)
    opt = FusedAdamW(params, **hp)
    _train_intermittent(opt, params, 3, dtype=dtype)
    sd = opt.state_dict()
    assert len({float(st["step"]) for st in sd["state"].values()}) > 1
    fresh = _params(98, dtype=dtype)
    with torch.no_grad():
        for p, q in zip(fresh, params):
            p.copy_(q)
    opt2 = FusedAdamW(fresh, **hp)
    opt2.load_state_dict(sd)
    _train_intermittent(opt2, fresh, 7, first=4, dtype=dtype)
    for p, q in zip(fresh, ref_params):
        assert torch.equal(p, q)
        for key in ("exp_avg", "exp_avg_sq", "max_exp_avg_sq"):
            assert torch.equal(opt2.state[p][key], ref.state[q][key])
        if dtype != torch.float32:
            assert torch.equal(opt2.state[p]["master_param"], ref.state[q]["master_param"])
    assert ([float(st["step"]) for st in opt2.state_dict()["state"].values()]
            == [float(st["step"]) for st in ref.state_dict()["state"].values()])


def test_param_group_added_after_construction():
    """A group added with add_param_group after two steps gets its own bucket and its
    own step counts: both groups follow the oracle, and both share the global clip."""
    first = _params(17, shapes=SHAPES[:3])
    later = _params(18, shapes=SHAPES[3:])
    opt = FusedAdamW(first, lr=1e-3, max_grad_norm=0.05)
    lib = oracle.lib()
    oo = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=1e-4, amsgrad=False,
              maximize=False)
    refs = [oracle.OracleAdamW(_host(p), oo, lib_=lib) for p in first + later]
    for step in range(1, 6):
        if step == 3:
            opt.add_param_group({"params": later, "lr": 2e-3})
            for r in refs[3:]:
                r.opts = dict(oo, lr=2e-3)
        params = first + (later if step >= 3 else [])
        grads = _grads(17, step)[:len(params)]
        _set_grads(params, grads)
        opt.step()
        allg = np.concatenate([g.numpy().reshape(-1) for g in grads])
        s, c = lib.gradient_stats(allg, "f32")
        _, norm, coef = lib.clip_decision(s, c, 0.05)
        assert abs(opt.last_report["grad_norm"] - norm) <= 1e-5 * norm
        for r, g in zip(refs, grads):
            r.step(g.numpy().reshape(-1), "f32", clip_coef=coef)
    torch.cuda.synchronize()
    for p, r in zip(first + later, refs):
        gate(_host(p), r.p, 1e-5, "p")
    steps = [int(float(st["step"])) for st in opt.state_dict()["state"].values()]
    assert steps == [5, 5, 5, 3, 3]


def test_group_on_several_devices_or_on_the_cpu_is_rejected():
    mixed = _params(19, shapes=SHAPES[:2])
    mixed.append(torch.nn.Parameter(torch.zeros(3)))  # on the CPU
    with pytest.raises(ValueError, match="one CUDA device"):
        FusedAdamW(mixed)
    with pytest.raises(ValueError, match="CUDA parameters"):
        FusedAdamW([torch.nn.Parameter(torch.zeros(3))])


def test_torch_lr_scheduler_drives_the_learning_rate():
    """A torch LR scheduler changes param_groups[...]["lr"] between steps; every fused
    step takes the group's current lr (each step vs the oracle with that lr)."""
    params = _params(20)
    opt = FusedAdamW(params, lr=1e-2, weight_decay=0.01)
    sched = torch.optim.lr_scheduler.LambdaLR(opt, lambda k: 0.5 ** k)
    lib = oracle.lib()
    oo = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=0.01, amsgrad=False,
              maximize=False)
    refs = [oracle.OracleAdamW(_host(p), oo, lib_=lib) for p in params]
    for step in range(1, 5):
        lr = opt.param_groups[0]["lr"]
        assert lr == pytest.approx(1e-2 * 0.5 ** (step - 1))
        grads = _grads(20, step)
        _set_grads(params, grads)
        opt.step()
        sched.step()
        for r, g in zip(refs, grads):
            r.opts = dict(oo, lr=lr)
            r.step(g.numpy().reshape(-1), "f32")
    torch.cuda.synchronize()
    for p, r in zip(params, refs):
        gate(_host(p), r.p, 1e-5, "p")


def lib_bits(t, name):
    """A gradient as the oracle takes it: FP32 values, or BF16 bit patterns."""
    if name == "f32":
        return _host(t)
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)


def test_replaced_gradients_are_gathered_into_the_bucket():
    params = _params(14)
    ref_params = _params(14)
    opt = FusedAdamW(params, lr=1e-3)
    ref = FusedAdamW(ref_params, lr=1e-3)
    for step in range(1, 4):
        grads = _grads(14, step)
        for p, g in zip(params, grads):      # new tensors, not views of the bucket
            p.grad = g.to(DEV).clone()
        _set_grads(ref_params, grads)        # written into the bucket views
        opt.step()
        ref.step()
    torch.cuda.synchronize()
    for p, q in zip(params, ref_params):
        assert torch.equal(p, q)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_decoder_full_size(dtype):
    """FusedAdamW as the benchmark runs it, at full size: the 1,195,991,040-parameter
    decoder in 199 tensors, global clip 1.0, the update gated on the device.  BF16:
    FP32 masters and moments, BF16 gradients, the BF16 copy written in the same pass.
    FP32: parameters, gradients and moments in FP32.  Gradients N(0, 1e-3).  Three calls,
    the second with one +Inf (skipped).  Each call: the report against the oracle's
    statistics over the whole gradient, the skip decision, and 40,000 sampled
    parameters plus every tensor's first and last element (parameters or masters, m, v
    along the trajectory; the BF16 copy bit for bit)."""
    import dataclasses
    from gpu_harness import check_model_copy, grad_bits_from_device
    from synthetic.configs import CONFIG5, decoder_bucket_shapes
    name = "bf16" if dtype == torch.bfloat16 else "f32"
    params = [torch.nn.Parameter(torch.zeros(shape, dtype=dtype, device=DEV))
              for _, shape in decoder_bucket_shapes()]
    opt = FusedAdamW(params, lr=1e-3, weight_decay=1e-4, eps=1e-5, max_grad_norm=1.0)
    b = opt._buckets[0]
    n = b.n
    assert n == 1_195_991_040 and b.offsets[-1] + params[-1].numel() == n
    w = dataclasses.replace(CONFIG5.scaled(n), calls=3, inf_call=2, grad_dtype=name)
    w.fill_params_device(b.master)
    ends = [o for o in b.offsets] + [o + p.numel() - 1 for o, p in zip(b.offsets, params)]
    rng = np.random.default_rng(21)
    idx = np.unique(np.concatenate([rng.integers(0, n, 40_000), ends, [w.inf_index()]]))
    idx_t = torch.as_tensor(idx, device=DEV)
    lib = oracle.lib()
    traj = oracle.OracleAdamW(w.params_host(idx), w.options(), lib_=lib)
    assert np.array_equal(b.master[idx_t].cpu().numpy(), w.params_host(idx))
    for call in range(1, 4):
        w.fill_grad_device(call, b.grad)
        gh = w.grad_host(call, idx)
        assert np.array_equal(grad_bits_from_device(b.grad[idx_t]), gh)
        s_or, c_or = lib.gradient_stats(grad_bits_from_device(b.grad), name, 1.0)
        skip_or, norm_or, coef_or = lib.clip_decision(s_or, c_or, 1.0)
        before = b.master[idx_t].cpu().numpy()
        opt.step()
        torch.cuda.synchronize()
        rep = opt.last_report
        assert rep["skipped"] == skip_or == (call == 2)
        assert rep["nonfinite"] == c_or
        if not skip_or:
            assert abs(rep["grad_norm"] - norm_or) <= 1e-5 * norm_or
            assert coef_or < 1.0
        traj.step(gh, name, 1.0, skip_update=skip_or, clip_coef=coef_or)
        master = b.master[idx_t].cpu().numpy()
        if skip_or:
            assert np.array_equal(master, before)
            continue
        gate(master, traj.p, 1e-5, f"call {call} master")
        gate(b.m[idx_t].cpu().numpy(), traj.state.m, 1e-5, f"call {call} m")
        gate(b.v[idx_t].cpu().numpy(), traj.state.v, 1e-5, f"call {call} v")
        if b.model is not None:
            check_model_copy(grad_bits_from_device(b.model[idx_t]), master,
                             traj.p.astype(np.float32), name, lib, f"call {call} model copy")
    assert set(b.steps) == {2} and traj.state.t == 2
