"""Seeded random launch configurations on the GPU against the CPU oracle:
every mode, role class, barrier variant, workload, participant count, payload
size, thread count, round count and counter start, bit for bit."""
import numpy as np
import pytest

import cns_inputs as ci
import oracle
from tests.gpu_helpers import from_dev_u32, to_dev_f32, to_dev_u32

pytestmark = pytest.mark.gpu

SOFT, HARD = 1, 0
AIV, AIC, MIX = 0, 1, 2
RING = [oracle.WL_RING_AFFINE, oracle.WL_RING_ROTATE, oracle.WL_XORSHIFT]


def configs(n, seed=2024):
    rng = np.random.RandomState(seed)
    out = []
    for i in range(n):
        mode = int(rng.choice([SOFT, HARD]))
        core = int(rng.choice([AIV, AIC, MIX]))
        variant = int(rng.randint(0, 6))
        ratio = int(rng.randint(1, 4)) if core == MIX else 0
        group = 1 + ratio if core == MIX else 1
        launch = int(rng.randint(1, 150 // group + 1))
        grid = launch * group
        used = int(rng.randint(1, grid + 1)) if (mode == SOFT and rng.rand() < 0.3) else 0
        P = used or grid
        wl = int(rng.choice(RING + [oracle.WL_JACOBI]))
        slots = int(rng.randint(0, 300))
        N = int(rng.randint(1, 60000))
        rounds = int(rng.randint(0, 120))
        threads = int(rng.choice([32, 64, 128, 256, 512]))
        near_wrap = rng.rand() < 0.25
        out.append(dict(mode=mode, core=core, variant=variant, ratio=ratio, launch=launch, grid=grid, used=used,
                        P=P, wl=wl, slots=slots, N=N, rounds=rounds, threads=threads, near_wrap=near_wrap,
                        seed=1000 + i))
    return out


@pytest.fixture(scope="module")
def cns():
    import torch
    import counted_notify_sync_gb300 as c
    c.build()
    torch.cuda.set_device(0)
    return c


@pytest.mark.parametrize("cfg", configs(96), ids=lambda c: f"m{c['mode']}c{c['core']}v{c['variant']}w{c['wl']}P{c['P']}")
def test_random_config(cns, cfg):
    import torch
    c = cfg
    ws = cns.new_workspace()
    # counter start: 0, or a few rounds before the wrap of the counter this path arrives on
    if c["near_wrap"]:
        if c["mode"] == SOFT:
            Pc = c["P"]
        else:
            Pc = None        # cluster size is chosen by the library: start at 0
        start = (oracle.counter_modulus(Pc) - 3 * Pc) if Pc else 0
        ws = cns.new_workspace(start_value=start)
    else:
        start = 0
    status = torch.zeros(c["grid"], dtype=torch.int32, device="cuda")
    if c["wl"] == oracle.WL_JACOBI:
        u0 = ci.jacobi_field(c["N"], seed=c["seed"])
        b0 = to_dev_f32(u0)
        b1 = torch.zeros_like(b0)
        d, rc = cns.run_syncall(c["mode"], c["core"], cns.CNS_WL_JACOBI, c["launch"], b0, b1, c["rounds"],
                                used_cores=c["used"], aiv_ratio=c["ratio"], elems=c["N"], threads=c["threads"],
                                workspace=ws, cta_status=status, variant=c["variant"])
        got = (b1 if c["rounds"] & 1 else b0).cpu().numpy()
        want, fc, orc = oracle.syncall_run_jacobi(u0, c["rounds"], c["P"], start if c["mode"] == SOFT else 0)
        np.testing.assert_array_equal(got, want)
    else:
        v0 = ci.ring_payload(c["seed"], c["P"], c["slots"])
        b0 = to_dev_u32(v0) if v0.size else None
        b1 = torch.zeros_like(b0) if v0.size else None
        d, rc = cns.run_syncall(c["mode"], c["core"], c["wl"], c["launch"], b0, b1, c["rounds"],
                                used_cores=c["used"], aiv_ratio=c["ratio"], elems=c["slots"], threads=c["threads"],
                                workspace=ws, cta_status=status, variant=c["variant"])
        want, fc, orc = oracle.syncall_run_ring(c["wl"], v0, c["rounds"], start if c["mode"] == SOFT else 0)
        if v0.size:
            got = from_dev_u32(b1 if c["rounds"] & 1 else b0).reshape(c["P"], c["slots"])
            np.testing.assert_array_equal(got, want)
    assert orc == oracle.OK and rc == 0 and d.device_status == 0
    assert d.participants == c["P"] and d.grid_ctas == c["grid"]
    if c["mode"] == SOFT:
        assert d.final_counter == fc
    else:
        clusters = c["grid"] // d.cluster_used
        assert d.final_counter == (c["rounds"] * clusters) % oracle.counter_modulus(clusters)
    st = status.cpu().numpy()
    assert ((st[:c["P"]] & 0xFF) == cns.CNS_CTA_DONE).all()
    assert ((st[c["P"]:] & 0xFF) == cns.CNS_CTA_IDLE).all()


def configs_more(n, seed=4242):
    """A second seeded batch over the later variants: the sense-flip counter
    (6), and arrival only (7, 8) which takes empty rounds only."""
    rng = np.random.RandomState(seed)
    out = []
    for i in range(n):
        mode = int(rng.choice([SOFT, HARD]))
        core = int(rng.choice([AIV, AIC, MIX]))
        variant = int(rng.choice([6, 7, 8]))
        ratio = int(rng.randint(1, 4)) if core == MIX else 0
        group = 1 + ratio if core == MIX else 1
        launch = int(rng.randint(1, 150 // group + 1))
        grid = launch * group
        used = int(rng.randint(1, grid + 1)) if (mode == SOFT and rng.rand() < 0.3) else 0
        P = used or grid
        wl = oracle.WL_EMPTY if variant in (7, 8) else int(rng.choice(RING + [oracle.WL_JACOBI]))
        slots = int(rng.randint(0, 300))
        N = int(rng.randint(1, 60000))
        rounds = int(rng.randint(0, 120))
        threads = int(rng.choice([32, 64, 128, 256, 512]))
        out.append(dict(mode=mode, core=core, variant=variant, ratio=ratio, launch=launch, grid=grid, used=used,
                        P=P, wl=wl, slots=slots, N=N, rounds=rounds, threads=threads, seed=5000 + i))
    return out


@pytest.mark.parametrize("cfg", configs_more(60), ids=lambda c: f"m{c['mode']}c{c['core']}v{c['variant']}w{c['wl']}P{c['P']}")
def test_random_config_later_variants(cns, cfg):
    import torch
    c = cfg
    ws = cns.new_workspace()
    status = torch.zeros(c["grid"], dtype=torch.int32, device="cuda")
    if c["wl"] == oracle.WL_EMPTY:
        d, rc = cns.run_syncall(c["mode"], c["core"], cns.CNS_WL_EMPTY, c["launch"], None, None, c["rounds"],
                                used_cores=c["used"], aiv_ratio=c["ratio"], threads=c["threads"], workspace=ws,
                                cta_status=status, variant=c["variant"])
        fc, orc = oracle.syncall_run_empty(c["P"], c["rounds"])
    elif c["wl"] == oracle.WL_JACOBI:
        u0 = ci.jacobi_field(c["N"], seed=c["seed"])
        b0 = to_dev_f32(u0)
        b1 = torch.zeros_like(b0)
        d, rc = cns.run_syncall(c["mode"], c["core"], cns.CNS_WL_JACOBI, c["launch"], b0, b1, c["rounds"],
                                used_cores=c["used"], aiv_ratio=c["ratio"], elems=c["N"], threads=c["threads"],
                                workspace=ws, cta_status=status, variant=c["variant"])
        got = (b1 if c["rounds"] & 1 else b0).cpu().numpy()
        want, fc, orc = oracle.syncall_run_jacobi(u0, c["rounds"], c["P"])
        np.testing.assert_array_equal(got, want)
    else:
        v0 = ci.ring_payload(c["seed"], c["P"], c["slots"])
        b0 = to_dev_u32(v0) if v0.size else None
        b1 = torch.zeros_like(b0) if v0.size else None
        d, rc = cns.run_syncall(c["mode"], c["core"], c["wl"], c["launch"], b0, b1, c["rounds"],
                                used_cores=c["used"], aiv_ratio=c["ratio"], elems=c["slots"], threads=c["threads"],
                                workspace=ws, cta_status=status, variant=c["variant"])
        want, fc, orc = oracle.syncall_run_ring(c["wl"], v0, c["rounds"])
        if v0.size:
            got = from_dev_u32(b1 if c["rounds"] & 1 else b0).reshape(c["P"], c["slots"])
            np.testing.assert_array_equal(got, want)
    assert orc == oracle.OK and rc == 0 and d.device_status == 0
    assert d.participants == c["P"] and d.grid_ctas == c["grid"]
    Pc = c["P"] if c["mode"] == SOFT else c["grid"] // d.cluster_used
    if c["variant"] == 6:
        assert d.final_counter == (c["rounds"] % 2) << 31
    else:
        assert d.final_counter == (c["rounds"] * Pc) % oracle.counter_modulus(Pc)
    st = status.cpu().numpy()
    assert ((st[:c["P"]] & 0xFF) == cns.CNS_CTA_DONE).all()
    assert ((st[c["P"]:] & 0xFF) == cns.CNS_CTA_IDLE).all()
