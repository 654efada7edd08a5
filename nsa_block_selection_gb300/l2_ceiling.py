"""The gather ceiling of the selection forward, measured on the GPU at hand.

The forward's hot step is the block gather ("[wave] NSA: selection attention
forward kernel", section "MI350 considerations"). With one KV group's K/V
resident in L2, its blocks reach the SMs from L2, not HBM, so HBM bandwidth
does not bound it. :func:`measure` times the library's probe kernel
(``nsa_probe_l2_gather``): every SM issues the forward's own TMA copies (16
keys x 64 dims, 128-byte swizzle, evict_last) for random blocks of the same
K/V and does nothing else. The best rate over a few in-flight depths is the
ceiling of the forward's gathered bytes per second.

``python -m nsa_block_selection_gb300.l2_ceiling`` runs the full sweep on
cuda:0 (depths, box sizes, layouts, active SMs, per-SM rates, the
workloads' own rows) and prints one JSON object; ``... l2_ceiling
ncu-case`` launches each measured kernel twice on the m16k_bs64 workload,
for a counter capture.
"""

from __future__ import annotations

import json
import statistics
import sys
import time

from . import _lib

# per-SM shared memory the probe's CTAs share (bytes), and the part the
# runtime reserves per CTA
SMEM_PER_SM = 228 * 1024
SMEM_RESERVED_PER_CTA = 1024
MAX_WARPS_PER_SM = 64

# (warps per CTA, CTAs per SM, tiles in flight per warp). The first is the
# forward's own depth: 4 warps x 4 CTAs per SM, a K and a V tile each
# (128 KB per SM in flight).
FORWARD_DEPTH = (4, 4, 2)
SWEEP = (
    (4, 4, 1), (8, 2, 1),                                     # 64 KB per SM
    FORWARD_DEPTH, (16, 1, 2), (32, 1, 1), (8, 2, 2),          # 128 KB
    (16, 2, 1), (8, 4, 1),
    (4, 4, 3), (8, 2, 3), (16, 1, 3), (4, 1, 12), (2, 4, 6),   # 192 KB
    (1, 16, 3), (8, 1, 6), (12, 2, 2), (24, 1, 2), (16, 3, 1), (8, 6, 1),
)
CEILING_SET = (FORWARD_DEPTH, (32, 1, 1), (16, 2, 1), (8, 4, 1), (16, 1, 2))
# depths for the index-driven probe (one launch moves a whole workload's tiles)
ROWS_SET = (FORWARD_DEPTH, (32, 1, 1), (16, 2, 1), (8, 4, 1), (16, 1, 2), (4, 4, 1),
            (8, 2, 2))


def smem_bytes(D, warps, slots, rows=16):
    """Dynamic shared memory of one probe CTA (as the library sizes it)."""
    return warps * slots * (D // 64) * rows * 128 + warps * slots * 8 + 1024


def fits(D, warps, ctas_per_sm, slots, rows=16):
    """Whether ctas_per_sm probe CTAs can be resident on one SM at once."""
    per = smem_bytes(D, warps, slots, rows) + SMEM_RESERVED_PER_CTA
    return (smem_bytes(D, warps, slots, rows) <= 227 * 1024 and ctas_per_sm * per <= SMEM_PER_SM
            and ctas_per_sm * warps <= MAX_WARPS_PER_SM and ctas_per_sm <= 32)


def run_once(k, v, g, bs, ctas, warps, slots, loads, seed=1, record=None, rows=16):
    """(bytes, ms) of one probe launch on torch's current stream, timed with
    CUDA events on that stream."""
    import torch

    st = torch.cuda.current_stream(k.device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    n = _lib.probe_l2_gather(k, v, g, bs, ctas, warps, slots, loads, seed, record=record,
                             stream=st, rows_per_box=rows)
    e1.record(st)
    e1.synchronize()
    rc = _lib.sync_status(st)
    if rc != 0:
        raise _lib.NsaError(rc, "nsa_probe_l2_gather (device wait)")
    return n, e0.elapsed_time(e1)


def time_config(k, v, g, bs, sms, cfg, seconds=0.25, sm_count=None, record=False,
                rate_hint=None):
    """Rate of one (warps, CTAs per SM, slots) configuration on ``sm_count``
    SMs' worth of CTAs (default: all): a short calibration launch (which
    also brings the K/V into L2), then one launch sized to last ``seconds``
    at the calibration's rate (or at ``rate_hint`` bytes/s, when given)."""
    import torch

    warps, cps, slots = cfg[:3]
    rows = cfg[3] if len(cfg) > 3 else 16
    D = k.shape[2]
    ctas = (sm_count or sms) * cps
    n, ms = run_once(k, v, g, bs, ctas, warps, slots, 64 * slots, rows=rows)
    rate = rate_hint or n / (ms * 1e-3)
    per_warp = max(16 * slots, int(rate * seconds / (ctas * warps * (D // 64) * rows * 128)))
    rec = torch.zeros((ctas, 3), dtype=torch.int64, device=k.device) if record else None
    n, ms = run_once(k, v, g, bs, ctas, warps, slots, per_warp, seed=7, record=rec, rows=rows)
    out = {"warps_per_cta": warps, "ctas_per_sm": cps, "slots_per_warp": slots,
           "rows_per_box": rows, "ctas": ctas,
           "inflight_kb_per_sm": cps * warps * slots * (D // 64) * rows * 128 // 1024,
           "bytes": n, "ms": ms, "gbs": n / (ms * 1e-3) / 1e9}
    if rec is not None:
        out["per_cta"] = rec.cpu()
    return out


def time_rows(k, v, idx, bs, sms, cfg, flush=None, reps=3, pad=0):
    """Mean ms of the index-driven probe over ``reps`` launches (after one
    untimed launch), each preceded by ``flush()`` outside the events;
    ``pad`` bytes of unused shared memory per CTA."""
    import torch

    warps, cps, slots = cfg
    st = torch.cuda.current_stream(k.device)
    ts = []
    for r in range(reps + 1):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        _lib.probe_gather_rows(k, v, idx, bs, sms * cps, warps, slots, stream=st,
                               extra_smem_bytes=pad)
        e1.record(st)
        e1.synchronize()
        if r:
            ts.append(e0.elapsed_time(e1))
    rc = _lib.sync_status(st)
    if rc != 0:
        raise _lib.NsaError(rc, "nsa_probe_gather_rows (device wait)")
    return statistics.mean(ts)


def measure(k, v, bs, g=0, idx=None, gathered_bytes=None, flush=None, seconds=0.25,
            long_seconds=2.0, configs=CEILING_SET, rows_configs=ROWS_SET, clocks=None):
    """The gather ceiling for K, V [B, N, G, D] (fp16).

    Random blocks of group g of batch 0: each configuration of ``configs``
    for ``seconds``, the best again for ``long_seconds`` (``clocks``, an
    object with start()/stop(), samples the SM clocks around that run).
    With ``idx`` (the workload's block_indices) and ``gathered_bytes`` (its
    gathered K/V bytes, as the forward's metric counts them), also the
    index-driven probe at each depth of ``rows_configs``: the forward's own
    copies alone, as gathered bytes per second. ``peak_gbs`` is the best rate
    of either."""
    import torch

    dev = k.device
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    D = k.shape[3]
    k0, v0 = k[0], v[0]
    rows = []
    for cfg in configs:
        if fits(D, *cfg):
            rows.append(time_config(k0, v0, g, bs, sms, cfg, seconds))
    best = max(rows, key=lambda r: r["gbs"])
    cfg = (best["warps_per_cta"], best["ctas_per_sm"], best["slots_per_warp"])
    if clocks is not None:
        clocks.start()
    final = time_config(k0, v0, g, bs, sms, cfg, long_seconds, rate_hint=best["gbs"] * 1e9)
    clk = clocks.stop() if clocks is not None else None
    fwd = next((r for r in rows if (r["warps_per_cta"], r["ctas_per_sm"],
                                   r["slots_per_warp"]) == FORWARD_DEPTH), None)
    out = {
        "random_blocks": {
            "peak_gbs": max(final["gbs"], best["gbs"]),
            "long_run": {k2: final[k2] for k2 in ("gbs", "ms", "bytes")},
            "best_config": list(cfg),
            "forward_depth_gbs": fwd["gbs"] if fwd else None,
            "configs": [[r["warps_per_cta"], r["ctas_per_sm"], r["slots_per_warp"],
                         round(r["gbs"], 1)] for r in rows],
            "clocks": clk,
            "pattern": f"TMA 16 keys x 64 dims boxes (128B swizzle, evict_last), K and V tiles "
                       f"alternating, random {bs}-key blocks of group {g} of K/V "
                       f"[{k0.shape[0]}, {k0.shape[1]}, {D}] fp16 "
                       f"({2 * k0.shape[0] * D * 2 / 1e6:.1f} MB in the group)"},
        "sms": sms,
        "config_key": "[warps per CTA, CTAs per SM, copies in flight per warp, GB/s]",
    }
    peak, src = out["random_blocks"]["peak_gbs"], "random_blocks"
    if idx is not None and gathered_bytes:
        rr = []
        for c in rows_configs:
            if fits(D, *c):
                ms = time_rows(k, v, idx, bs, sms, c, flush)
                rr.append([c[0], c[1], c[2], round(gathered_bytes / (ms * 1e-3) / 1e9, 1),
                           round(ms, 4)])
        rb = max(rr, key=lambda r: r[3])
        out["workload_rows"] = {
            "peak_gbs": rb[3], "best_config": rb[:3], "best_ms": rb[4],
            "forward_depth_gbs": next((r[3] for r in rr if tuple(r[:3]) == FORWARD_DEPTH),
                                      None),
            "configs": rr,
            "pattern": "the forward's own TMA copies for the workload's index rows (every "
                       "16-key tile it gathers, K then V), no computation; L2 flushed before "
                       "each launch; rate = the metric's gathered bytes / time"}
        if rb[3] > peak:
            peak, src = rb[3], "workload_rows"
    out["peak_gbs"] = peak
    out["peak_from"] = src
    return out


def per_sm_summary(per_cta, sms):
    """Rates per SM from per-CTA (SM id, start, end) records of one launch:
    bytes are equal per CTA, so an SM's rate is its CTAs' count over their
    span. Returns min / median / max over SMs and the mean of the SMs with
    ids below and above sms / 2."""
    import collections

    spans = collections.defaultdict(list)
    for smid, t0, t1 in per_cta.tolist():
        spans[int(smid)].append((t0, t1))
    rate = {}
    for smid, sp in spans.items():
        t0 = min(a for a, _ in sp)
        t1 = max(b for _, b in sp)
        rate[smid] = len(sp) / max(t1 - t0, 1)
    vals = sorted(rate.values())
    lo = [r for s, r in rate.items() if s < sms // 2]
    hi = [r for s, r in rate.items() if s >= sms // 2]
    starts = [a for sp in spans.values() for a, _ in sp]
    norm = statistics.median(vals)
    return {"sms_seen": len(rate), "min_rel": vals[0] / norm, "max_rel": vals[-1] / norm,
            "low_ids_rel": statistics.mean(lo) / norm if lo else None,
            "high_ids_rel": statistics.mean(hi) / norm if hi else None,
            "start_spread_us": (max(starts) - min(starts)) / 1e3}


def sweep(seconds=0.25):
    """The full sweep on cuda:0 (for the committed profile summary)."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    gen = torch.Generator(device=dev).manual_seed(3)

    def kv(N, G, D=128):
        return (torch.randn((N, G, D), generator=gen, device=dev).half(),
                torch.randn((N, G, D), generator=gen, device=dev).half())

    out = {"device": torch.cuda.get_device_name(dev), "sms": sms, "seconds_per_config": seconds}
    # 1. in-flight depth, the forward's layout: one group of [65536, 8, 128]
    k, v = kv(65536, 8)
    out["depth"] = [time_config(k, v, 0, 64, sms, c, seconds) for c in SWEEP
                    if fits(128, *c)]
    for r in out["depth"]:
        r.pop("per_cta", None)
    # 2. per-SM rates at the forward's depth (SM ids, both halves)
    r = time_config(k, v, 0, 64, sms, FORWARD_DEPTH, seconds, record=True)
    out["per_sm_forward_depth"] = per_sm_summary(r.pop("per_cta"), sms)
    out["per_sm_forward_depth"]["gbs"] = r["gbs"]
    # 3. active SMs: the same depth on fewer SMs
    out["active_sms"] = []
    for n in (sms // 4, sms // 2, 3 * sms // 4, sms):
        r = time_config(k, v, 0, 64, sms, FORWARD_DEPTH, seconds, sm_count=n)
        out["active_sms"].append({"sms": n, "gbs": r["gbs"], "gbs_per_sm": r["gbs"] / n})
    best_cfg = max(out["depth"], key=lambda r: r["gbs"])
    bc = (best_cfg["warps_per_cta"], best_cfg["ctas_per_sm"], best_cfg["slots_per_warp"])
    out["active_sms_best"] = []
    for n in (sms // 4, sms // 2, 3 * sms // 4, sms):
        r = time_config(k, v, 0, 64, sms, bc, seconds, sm_count=n)
        out["active_sms_best"].append({"config": list(bc), "sms": n, "gbs": r["gbs"],
                                       "gbs_per_sm": r["gbs"] / n})
    # 4. layouts with the same 33.5 MB: the strided group (2 KB key stride),
    # a contiguous [65536, 1, 128] pair, all 8 groups of [8192, 8, 128]
    lay = []
    for name, N, G, g in (("one group of [65536, 8, 128] (2 KB key stride)", 65536, 8, 0),
                          ("contiguous [65536, 1, 128] (256 B key stride)", 65536, 1, 0),
                          ("all groups of [8192, 8, 128], group drawn per block", 8192, 8, -1)):
        del k, v
        k, v = kv(N, G)
        for cfg in (FORWARD_DEPTH, bc):
            r = time_config(k, v, g, 64, sms, cfg, seconds)
            lay.append({"layout": name, "config": list(cfg), "gbs": r["gbs"]})
    out["layouts"] = lay
    # 5. block size 32
    del k, v
    k, v = kv(65536, 8)
    out["bs32"] = [{"config": list(c), "gbs": time_config(k, v, 0, 32, sms, c, seconds)["gbs"]}
                   for c in (FORWARD_DEPTH, bc)]
    # 6. larger boxes (32 or 64 key rows per TMA copy), up to 128 KB per SM
    out["box_rows"] = []
    for c in ((4, 4, 2, 16), (32, 1, 1, 16), (4, 4, 1, 32), (8, 2, 1, 32), (16, 1, 1, 32),
              (2, 4, 2, 32), (4, 2, 1, 64), (8, 1, 1, 64), (2, 4, 1, 64), (1, 8, 1, 64)):
        if fits(128, *c):
            r = time_config(k, v, 0, 64, sms, c, seconds)
            out["box_rows"].append([*c, round(r["gbs"], 1)])
    del k, v
    # 7. the workloads' own rows (index-driven probe), every depth
    from . import inputs as ginp
    from .metrics import count_work

    flush_buf = torch.empty(512 << 18, dtype=torch.float32, device=dev)
    out["workload_rows"] = {}
    for name in ("m64k_bs64", "m32k_bs32"):
        w = ginp.workload(name)
        idx = torch.from_numpy(ginp.make_block_indices(w, ginp.default_seed(name))).to(dev)
        kk = torch.randn((w.B, w.N, w.G, w.D), generator=gen, device=dev).half()
        vv = torch.randn((w.B, w.N, w.G, w.D), generator=gen, device=dev).half()
        nbytes = count_work(idx, w.N, w.block_size, w.heads_per_group, w.D)["gathered_bytes"]
        rr = []
        for c in SWEEP:
            if fits(w.D, *c):
                ms = time_rows(kk, vv, idx, w.block_size, sms, c, lambda: flush_buf.fill_(1.0))
                rr.append([c[0], c[1], c[2], round(nbytes / (ms * 1e-3) / 1e9, 1), round(ms, 4)])
        out["workload_rows"][name] = {"gathered_bytes": nbytes, "configs": rr}
        if name == "m64k_bs64":
            # the forward's depth with unused shared memory added per CTA:
            # where the rate falls off as a kernel reserves more
            pads = []
            for pad_kb in (0, 8, 12, 16, 20, 24, 28, 32, 40, 48):
                ms = time_rows(kk, vv, idx, w.block_size, sms, FORWARD_DEPTH,
                               lambda: flush_buf.fill_(1.0), pad=pad_kb * 1024)
                pads.append([pad_kb, (smem_bytes(w.D, 4, 2) + pad_kb * 1024) * 4 // 1024,
                             round(nbytes / (ms * 1e-3) / 1e9, 1)])
            out["workload_rows"][name]["smem_pad"] = pads
        del idx, kk, vv
    return out


def ncu_case(name="m16k_bs64"):
    """One launch each, after one untimed launch each, of: the forward on the
    workload, the index-driven probe on its rows (the forward's depth), and
    the random-block probe (32 warps per SM, one copy each) on group 0 of
    the workload's K/V and on a contiguous [N, 1, 128] pair of the same
    size -- the case the committed L2 counter summary is captured on."""
    import torch

    from . import inputs as ginp
    from ._lib import sel_attn_fwd

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    w = ginp.workload(name)
    q, k, v, idx = (torch.from_numpy(x).to(dev) for x in ginp.make_inputs(w))
    gen = torch.Generator(device=dev).manual_seed(3)
    kc = torch.randn((w.N, 1, w.D), generator=gen, device=dev).half()
    vc = torch.randn((w.N, 1, w.D), generator=gen, device=dev).half()
    ks, vs = k[0], v[0]
    loads = 4000
    for _ in range(2):  # untimed launch of each, then the one ncu captures
        sel_attn_fwd(q, k, v, idx, w.block_size)
        _lib.probe_gather_rows(k, v, idx, w.block_size, sms * 4, 4, 2)
        _lib.probe_l2_gather(ks, vs, 0, w.block_size, sms, 32, 1, loads)
        _lib.probe_l2_gather(kc, vc, 0, w.block_size, sms, 32, 1, loads)
        torch.cuda.synchronize()
    assert _lib.sync_status() == 0
    print(f"ncu case {name}: forward, rows probe (4, 4, 2), random probe (32, 1, 1) on "
          f"group 0 and on a contiguous [{w.N}, 1, {w.D}] pair; each launched twice")


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    if argv and argv[0] == "ncu-case":
        ncu_case(argv[1] if len(argv) > 1 else "m16k_bs64")
        return 0
    seconds = float(argv[0]) if argv else 0.25
    t0 = time.time()
    res = sweep(seconds)
    res["wall_s"] = time.time() - t0
    print(json.dumps(res, indent=1))
    return 0


if __name__ == "__main__":
    sys.exit(main())
