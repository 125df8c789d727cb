"""Benchmark of the image-VAE decoder hot path on GB300.

One step = one whole decode of a 1024^2 frame by the Qwen-Image-2.1-style
(Wan RMS_norm, DupUp) decoder: latent [16,128,128] -> RGB [3,1024,1024],
random He-normal f16 weights, synthetic latent N(mu_c, sigma_c) per channel.
Every step runs every hot-path stage: the implicit-GEMM 3x3 convs with the
nearest-2x fold and fused bias/residual/DupUp epilogues, RMS_norm, the
guarded casts, the 1x1 convs, the fused mid attention, conv_out to NCHW.

value   = algorithmic FLOPs of one decode (2*M*N*K over all convs with real
          channels + the attention's 4*m^2*c) x frames / timed seconds, TFLOP/s
e2e     = the same through the host-buffer C-ABI call (latent copied in from
          pinned host memory, RGB copied out, inside the timed region)
roofline: the 3x3 conv launches at the 1024^2 stage (M = 1048576, N = 144,
          K = 1296), timed with CUDA events on the launching stream inside the
          timed region, against the measured burst dense bf16 peak (f16 runs at
          the bf16 rate on the tensor pipe; the conv runs at the maximum SM
          clock inside a ~14 ms step, as the burst measurement does); the
          fractions of the sustained and of the nominal 2.25 PFLOP/s rate are
          reported beside it.

``--impl reference`` times the CPU oracle (float64 numpy) instead, on a
bounded sample of the same workload: the same decoder on a 16x16 latent.
Under torchrun (N > 1) every rank decodes its own frame (independent
replicas, no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "3×3 implicit-GEMM conv TFLOP/s (frac of f16 peak); VAE decode ms/frame at 1024²"
LATENT = (16, 128, 128)
WORKLOAD = ("Qwen-Image-2.1-style decoder (RMS_norm, DupUp; widths 1152/576/288/144, 3 ResNets per block), "
            "latent [16,128,128] -> RGB [3,1024,1024]")
DOMINANT = {"h": 1024, "w": 1024, "cin": 144, "cout": 144}
NOMINAL_F16_TFLOPS = 2250.0  # GB300 dense f16/bf16 tensor rate, datasheet (no sparsity)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops_sustained"]), float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1700.0, 1900.0, 6800.0, "fallback"


def decoder_flops(dec, h0, w0):
    """Algorithmic FLOPs of one decode, from the description's shapes."""
    conv = 0.0
    h, w = h0, w0

    def c(cv, hh, ww):
        return 2.0 * hh * ww * cv.cout * cv.cin * cv.k * cv.k

    if dec.post_quant is not None:
        conv += c(dec.post_quant, h, w)
    conv += c(dec.conv_in, h, w)
    for r in (dec.mid_res1, dec.mid_res2):
        conv += c(r.conv1, h, w) + c(r.conv2, h, w) + (c(r.shortcut, h, w) if r.shortcut is not None else 0)
    m, ch = h * w, dec.mid_attn.c
    attn = 4.0 * m * m * ch + 4 * 2.0 * m * ch * ch
    for u in dec.ups:
        for r in u.resnets:
            conv += c(r.conv1, h, w) + c(r.conv2, h, w) + (c(r.shortcut, h, w) if r.shortcut is not None else 0)
        if u.up is not None:
            h, w = 2 * h, 2 * w
            conv += c(u.up, h, w)
    conv += c(dec.conv_out, h, w)
    return conv, attn


def clock_sampler_start(path):
    try:
        f = open(path, "w")
        p = subprocess.Popen(["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,"
                              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                              "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "200"],
                             stdout=f, stderr=subprocess.DEVNULL)
        return p, f
    except Exception:
        return None, None


def clock_sampler_stop(p, f, path, gpu_index):
    if p is None:
        return None
    p.terminate()
    try:
        p.wait(timeout=5)
    except Exception:
        p.kill()
    f.close()
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in open(path):
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9 or parts[0] != str(gpu_index):
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    load = [s for s in sm if s > 0.5 * max(sm)] or sm
    return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm)}


def kernel_source_hash() -> str:
    """sha256 over the conv kernel's sources (csrc/vae_conv.cu, vae_common.cuh,
    vae_conv.h, in that order) with C++ comments and blank space removed, so
    that edits to comments alone keep a capture valid."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("vae_conv.cu", "vae_common.cuh", "vae_conv.h"):
        src = open(os.path.join(ROOT, "implicit_gemm_convolution_vae_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()


def traffic_from_profiles():
    """DRAM bytes per launch of the dominant conv from the committed ncu summary,
    if it was taken on the current kernel source (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "conv3x3_1024x1024_144to144_ncu.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def cpu_oracle_sample(dec, seed=0, h0=16, w0=16, steps=1, warmup=0):
    import oracle
    from vae_inputs import latent_channel_stats
    z = latent_channel_stats(seed, 16, h0, w0)
    conv, attn = decoder_flops(dec, h0, w0)
    for _ in range(warmup):
        oracle.decode_rms(dec, z)
    ts = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.decode_rms(dec, z)
        ts.append(time.perf_counter() - t0)
    return conv + attn, ts


def cores_used():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("internal_api") in ("openblas", "mkl", "blis")]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def reduce_max(x: float, dist) -> float:
    """The maximum of x over all ranks (x itself without a process group): the
    job's time is its slowest rank's."""
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_unit: float, units_per_rank: int, world: int, seconds: float) -> float:
    """Throughput of the whole job: the units every rank processed over the slowest rank's time."""
    return flops_per_unit * units_per_rank * world / seconds / 1e12


def run_reference(args, rank):
    if rank != 0:
        return
    from vae_inputs import qwen_decoder
    dec = qwen_decoder(seed=0)
    flops, ts = cpu_oracle_sample(dec, steps=args.steps, warmup=args.warmup)
    tot = sum(ts)
    val = flops * len(ts) / tot / 1e12
    sample = "oracle (float64 numpy) decode of the same decoder on a 16x16 latent (128^2 frame), one per step"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(ts),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD + " (CPU oracle sample: latent [16,16,16])", "parallelism": "none"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_kernel(args):
    """One kernel at one shape, timed with CUDA events (for ncu captures and sweeps)."""
    import torch
    import implicit_gemm_convolution_vae_gb300 as vg
    vg.build()
    torch.manual_seed(0)
    vals = [int(v) for v in args.shape.split(",")]
    stream = torch.cuda.current_stream()
    if args.kernel in ("conv3d", "upconv3d"):
        # 3x3x3 causal conv over frames; upconv3d folds the spatial and temporal 2x
        f, h, w, cin, cout = vals
        up = args.kernel == "upconv3d"
        x = torch.randn(1, f, h, w, cin, device="cuda").half()
        wt = (torch.randn(cout, 3, 3, 3, cin, device="cuda") / (27 * cin) ** 0.5).half()
        b = torch.randn(cout, device="cuda") * 0.1
        Fo, H, W = (2 * f - 1, 2 * h, 2 * w) if up else (f, h, w)
        y = torch.empty(1, Fo, H, W, cout, device="cuda")
        if args.residual:
            y.normal_()  # the residual is the output itself: the in-place stream update
        fn = lambda: vg.conv3d_causal_ndhwc(x, wt, b, residual=y if args.residual else None, out=y, upsample=up,
                                            t_upsample=up)
        flops = 2.0 * Fo * H * W * cout * 27 * cin
        nbytes = x.numel() * 2 + y.numel() * 4 * (2 if args.residual else 1)
        h = w = 0
    else:
        h, w, cin, cout = vals
    if h == 0:
        pass
    elif args.kernel in ("conv3x3", "upconv3x3", "downconv3x3"):
        up = args.kernel == "upconv3x3"
        down = args.kernel == "downconv3x3"  # the encoder's far-side-padded stride-2 conv
        x = torch.randn(1, h, w, cin, device="cuda").half()
        wt = (torch.randn(cout, 3, 3, cin, device="cuda") / (9 * cin) ** 0.5).half()
        b = torch.randn(cout, device="cuda") * 0.1
        H, W = (2 * h, 2 * w) if up else ((h // 2, w // 2) if down else (h, w))
        y = torch.empty(1, H, W, cout, device="cuda")
        res = None
        if args.residual:
            y.normal_()  # the residual is the output itself: the in-place stream update
            res = y
        if args.subpixel and up:  # the sub-pixel form, credited at the 9-tap FLOP count
            wsub = vg.pack_subpixel_weights(wt)
            fn = lambda: vg.conv3x3_nhwc(x, wsub, b, residual=res, out=y, upsample=True, subpixel=True)
        else:
            fn = lambda: vg.conv3x3_nhwc(x, wt, b, residual=res, out=y, upsample=up, down=down,
                                         reflect=args.reflect or down)
        flops = 2.0 * H * W * cout * 9 * cin
        nbytes = x.numel() * 2 + y.numel() * 4 * (2 if args.residual else 1)
    elif args.kernel == "rmsnorm":
        x = torch.randn(h * w, cin, device="cuda")
        g = torch.ones(cin, device="cuda")
        y = torch.empty(h * w, cin, dtype=torch.float16, device="cuda")
        fn = lambda: vg.rmsnorm_silu(x, g, silu=True, out=y)
        flops, nbytes = 0.0, x.numel() * 6
    elif args.kernel == "conv3x3rms":
        # a ResNet's first conv with its second RMS_norm(+SiLU) in the epilogue (f16 rows only)
        x = torch.randn(1, h, w, cin, device="cuda").half()
        wt = (torch.randn(cout, 3, 3, cin, device="cuda") / (9 * cin) ** 0.5).half()
        b = torch.randn(cout, device="cuda") * 0.1
        g = torch.ones(cout, device="cuda")
        yn = torch.empty(1, h, w, cout, dtype=torch.float16, device="cuda")
        fn = lambda: vg.conv3x3_nhwc_rms(x, wt, g, b, out=yn, silu=True)
        flops = 2.0 * h * w * cout * 9 * cin
        nbytes = x.numel() * 2 + yn.numel() * 2
    elif args.kernel in ("convgn", "convgn_fused"):
        # a 3x3 conv (f32 out, in-place residual) followed by GroupNorm(32)+SiLU -> f16:
        # convgn = conv + the standalone two-pass GroupNorm; convgn_fused = the conv
        # taking the statistics in its epilogue + the one-read apply
        x = torch.randn(1, h, w, cin, device="cuda").half()
        wt = (torch.randn(cout, 3, 3, cin, device="cuda") / (9 * cin) ** 0.5).half()
        b = torch.randn(cout, device="cuda") * 0.1
        y = torch.randn(1, h, w, cout, device="cuda")
        g = torch.ones(cout, device="cuda")
        bb = torch.zeros(cout, device="cuda")
        yn = torch.empty(1, h * w, cout, dtype=torch.float16, device="cuda")
        refl = args.reflect
        if args.kernel == "convgn":
            wsp = torch.empty(vg.groupnorm_workspace_bytes(1, h * w, cout, 32), dtype=torch.uint8, device="cuda")

            def fn():
                vg.conv3x3_nhwc(x, wt, b, residual=y, out=y, reflect=refl)
                vg.groupnorm_silu(y.reshape(1, h * w, cout), 32, g, bb, silu=True, out=yn, workspace=wsp)
        else:
            wsp = torch.empty(vg.conv3x3_gn_workspace_bytes(1, h, w, cout, 32, vg.PAD_REFLECT if refl else 0),
                              dtype=torch.uint8, device="cuda")

            def fn():
                _, st = vg.conv3x3_nhwc_gn(x, wt, 32, b, residual=y, out=y, reflect=refl, workspace=wsp)
                vg.groupnorm_apply(y.reshape(1, h * w, cout), 32, st, g, bb, silu=True, out=yn)
        flops = 2.0 * h * w * cout * 9 * cin
        nbytes = x.numel() * 2 + y.numel() * 4 * 2 + y.numel() * (4 + 2)
    elif args.kernel == "groupnorm":
        x = torch.randn(1, h * w, cin, device="cuda")
        g = torch.ones(cin, device="cuda")
        bb = torch.zeros(cin, device="cuda")
        y = torch.empty(1, h * w, cin, dtype=torch.float16, device="cuda")
        wsp = torch.empty(vg.groupnorm_workspace_bytes(1, h * w, cin, 32), dtype=torch.uint8, device="cuda")
        fn = lambda: vg.groupnorm_silu(x, 32, g, bb, silu=True, out=y, workspace=wsp)
        flops, nbytes = 0.0, x.numel() * 10
    elif args.kernel == "attention":
        m, c = h * w, cin
        x = torch.randn(m, c, device="cuda")
        ws_ = [(torch.randn(c, c, device="cuda") / c ** 0.5).half() for _ in range(4)]
        bs = [torch.randn(c, device="cuda") * 0.1 for _ in range(4)]
        g = torch.ones(c, device="cuda")
        wsp = torch.empty(vg.mid_attention_workspace_bytes(m, c), dtype=torch.uint8, device="cuda")
        fn = lambda: vg.mid_attention(x, vg.NORM_RMS, g, None, ws_[0], bs[0], ws_[1], bs[1], ws_[2], bs[2],
                                      ws_[3], bs[3], workspace=wsp)
        flops, nbytes = 4.0 * m * m * c + 8.0 * m * c * c, 0.0
    else:
        raise SystemExit(f"unknown kernel {args.kernel}")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(max(args.warmup, 1)):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    vg.sync_status()
    ms = statistics.median(ts)
    sust, burst, hbm, src = peaks()
    out = {"kernel": args.kernel, "shape": args.shape, "ms": ms, "steps": args.steps}
    if flops:
        out["tflops"] = flops / ms / 1e9
        out["frac_burst"] = out["tflops"] / burst
    if nbytes:
        out["gbs"] = nbytes / ms / 1e6
        out["frac_hbm"] = out["gbs"] / hbm
    print(json.dumps(out), flush=True)


def _event_ms(fn, reps, warmup=2):
    """Median-free mean of `reps` back-to-back calls, CUDA events on the current stream."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def weight_bytes(dec):
    """Device bytes of a decoder description's weights as the library stores them
    (f16 convs, f32 biases and norm parameters)."""
    tot = 0

    def conv(c):
        return 0 if c is None else c.w.size * 2 + (0 if c.b is None else c.b.size * 4)

    def norm(n):
        return n.gamma.size * 4 + (0 if getattr(n, "beta", None) is None else n.beta.size * 4)

    def res(r):
        return norm(r.norm1) + conv(r.conv1) + norm(r.norm2) + conv(r.conv2) + conv(r.shortcut)

    tot += conv(getattr(dec, "post_quant", None)) + conv(dec.conv_in) + res(dec.mid_res1) + res(dec.mid_res2)
    a = dec.mid_attn
    tot += norm(a.norm) + conv(a.q) + conv(a.k) + conv(a.v) + conv(a.o)
    for u in dec.ups:
        tot += sum(res(r) for r in u.resnets) + conv(u.up)
    return tot + norm(dec.norm_out) + conv(dec.conv_out)


def extra_configs(D, dec, reps=5):
    """The other configurations of the hot path, each timed on the device with CUDA
    events (inputs resident; reported beside the contract's number, not in it):
    the single 3x3 conv 32x32x64->64 (zero pad, nearest-2x fold from 16x16,
    replicate pad), the GroupNorm up block at 128^2 x 256, the FLUX-class decoder
    at 256^2, and the 1024^2 decoder at 2048^2 and 1536x2752, whole frame and in
    three bands from up block 2, with the decode's device memory."""
    import torch
    import implicit_gemm_convolution_vae_gb300 as vg
    from vae_inputs import (conv_case, flux_decoder, gn_up_block, latent_channel_stats, latent_normal,
                            stream_normal)
    out = {}
    # single conv, 75.5 MFLOP each
    c1 = conv_case(seed=0, n=1, h=32, w=32, cin=64, cout=64, name="bench.cfg1")
    x = torch.from_numpy(c1["x"]).cuda()
    xs = x[:, :16, :16, :].contiguous()
    w = torch.from_numpy(vg.pack_conv3x3(c1["w"])).cuda()
    b = torch.from_numpy(c1["b"]).cuda()
    y = torch.empty(1, 32, 32, 64, device="cuda")
    fl = 2.0 * 32 * 32 * 64 * 9 * 64
    for name, kw, xin in (("1a_zero_pad", {}, x), ("1b_upsample2x", {"upsample": True}, xs),
                          ("1c_replicate", {"replicate": True}, x)):
        ms = _event_ms(lambda: vg.conv3x3_nhwc(xin, w, b, out=y, **kw), 200, 20)
        out[f"conv3x3_cfg{name}"] = {"us": 1e3 * ms, "tflops": fl / ms / 1e9}
    # config 2: two GroupNorm ResNets(256) + nearest-2x + conv 256->256, at 128^2
    blk = gn_up_block(seed=0, c=256, nres=2)
    xs0 = torch.from_numpy(stream_normal(0, "cfg2.x", (128, 128, 256))).cuda().reshape(1, 128 * 128, 256)
    xd = xs0.clone()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    prm = [(dev(r.norm1.gamma), dev(r.norm1.beta), dev(vg.pack_conv3x3(r.conv1.w)), dev(r.conv1.b),
            dev(r.norm2.gamma), dev(r.norm2.beta), dev(vg.pack_conv3x3(r.conv2.w)), dev(r.conv2.b))
           for r in blk.resnets]
    wu, bu = dev(vg.pack_conv3x3(blk.up.w)), dev(blk.up.b)
    xn = torch.empty(1, 128 * 128, 256, dtype=torch.float16, device="cuda")
    hbuf = torch.empty(1, 128, 128, 256, device="cuda")
    xsf = torch.empty(1, 128 * 128, 256, dtype=torch.float16, device="cuda")
    yu = torch.empty(1, 256, 256, 256, device="cuda")
    gws = torch.empty(vg.groupnorm_workspace_bytes(1, 128 * 128, 256, 32), dtype=torch.uint8, device="cuda")

    def up_block():
        for g1, b1, w1, c1b, g2, b2, w2, c2b in prm:
            vg.groupnorm_silu(xd, 32, g1, b1, silu=True, out=xn, workspace=gws)
            vg.conv3x3_nhwc(xn.reshape(1, 128, 128, 256), w1, c1b, out=hbuf)
            vg.groupnorm_silu(hbuf.reshape(1, -1, 256), 32, g2, b2, silu=True, out=xn, workspace=gws)
            vg.conv3x3_nhwc(xn.reshape(1, 128, 128, 256), w2, c2b, residual=xd.reshape(1, 128, 128, 256),
                            out=xd.reshape(1, 128, 128, 256))
        vg.cast_f16(xd, 256, scale=2.0 ** -8, out=xsf)
        vg.conv3x3_nhwc(xsf.reshape(1, 128, 128, 256), wu, bu, upsample=True, oscale=256.0, out=yu)

    ms = _event_ms(up_block, 20, 3)
    fl2 = 4 * 2.0 * 128 * 128 * 256 * 9 * 256 + 2.0 * 256 * 256 * 256 * 9 * 256
    out["up_block_cfg2_128x128x256"] = {"ms": ms, "conv_tflops_effective": fl2 / ms / 1e9}
    # config 3: FLUX-class decoder, latent [16,32,32] -> 256^2
    fdec = flux_decoder(seed=0)
    FD = vg.Decoder(fdec)
    zf = torch.from_numpy(latent_normal(0, 16, 32, 32)).cuda()
    of = torch.empty(3, 256, 256, device="cuda")
    wsf = torch.empty(FD.workspace_bytes(32, 32), dtype=torch.uint8, device="cuda")
    ms = _event_ms(lambda: FD.decode(zf, out=of, workspace=wsf), 20, 3)
    cf, af = decoder_flops(fdec, 32, 32)
    out["flux_decoder_cfg3_256"] = {"ms_per_frame": ms, "tflops": (cf + af) / ms / 1e9,
                                    "mp_per_s": 256 * 256 / ms / 1e3}
    FD.close()
    del wsf
    # config 5: the 1024^2 decoder at 2048^2 and 1536x2752, whole and 3 bands from up block 2
    wb = weight_bytes(dec)
    for h0, w0 in ((256, 256), (192, 344)):
        z = torch.from_numpy(latent_channel_stats(5, 16, h0, w0)).cuda()
        o = torch.empty(3, 8 * h0, 8 * w0, device="cuda")
        cf, af = decoder_flops(dec, h0, w0)
        for label, opts in (("whole", None), ("3bands_from_block2", vg.Decoder.opts(band_from=2, nbands=3))):
            nb = D.workspace_bytes(h0, w0, opts)
            torch.cuda.synchronize()
            torch.cuda.reset_peak_memory_stats()
            base = torch.cuda.memory_allocated()
            ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
            ms = _event_ms(lambda: D.decode(z, out=o, opts=opts, workspace=ws), reps, 2)
            peak = torch.cuda.max_memory_allocated() - base
            out[f"qwen_decoder_{8 * h0}x{8 * w0}_{label}"] = {
                "ms_per_frame": ms, "mp_per_s": 64 * h0 * w0 / ms / 1e3, "tflops": (cf + af) / ms / 1e9,
                "workspace_bytes": nb,
                "device_bytes": nb + z.numel() * 4 + o.numel() * 4 + wb,
                "device_bytes_note": "workspace + latent + RGB output + weights (the decode allocates nothing else)",
                "torch_peak_allocated_bytes_during_decodes": int(peak)}
            del ws
        vg.sync_status()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip the other configurations (single convs, up block, FLUX decoder, 2048^2 frames)")
    ap.add_argument("--kernel", default=None,
                    help="time one kernel instead: conv3x3, upconv3x3, downconv3x3, conv3x3rms, conv3d, upconv3d, convgn, "
                         "convgn_fused, "
                         "rmsnorm, groupnorm, "
                         "attention")
    ap.add_argument("--shape", default="1024,1024,144,144",
                    help="h,w,cin,cout (attention: h,w,c,c; conv3d/upconv3d: f,h,w,cin,cout)")
    ap.add_argument("--residual", action="store_true")
    ap.add_argument("--subpixel", action="store_true", help="upconv3x3 in the sub-pixel form")
    ap.add_argument("--reflect", action="store_true", help="conv3x3 with reflect padding (the encoder's)")
    args = ap.parse_args()
    if args.kernel:
        return run_kernel(args)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank)
    args.warmup = max(args.warmup, 3)

    import torch
    import implicit_gemm_convolution_vae_gb300 as vg
    from vae_inputs import latent_channel_stats, qwen_decoder

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    vg.build()
    dec = qwen_decoder(seed=0)
    D = vg.Decoder(dec)
    h0, w0 = LATENT[1], LATENT[2]
    z = torch.from_numpy(latent_channel_stats(rank, *LATENT)).cuda()
    out = torch.empty((3, h0 * 8, w0 * 8), dtype=torch.float32, device="cuda")
    # The timed decodes carry CUDA events only around the full-resolution ResNet
    # convs (the roofline's kernel); every stage is timed in a separate decode.
    opts = vg.Decoder.opts(profile="fullres")
    opts_all = vg.Decoder.opts(profile=True)
    ws = torch.empty(D.workspace_bytes(h0, w0, opts), dtype=torch.uint8, device="cuda")
    conv_f, attn_f = decoder_flops(dec, h0, w0)
    step_flops = conv_f + attn_f
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        D.decode(z, out=out, opts=opts, workspace=ws)
    vg.sync_status()
    D.profile()  # drop warm-up records

    clk_path = os.path.join(tempfile.gettempdir(), f"vae_clocks_{os.getpid()}.csv")
    cp, cf = clock_sampler_start(clk_path)
    time.sleep(0.5)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        D.decode(z, out=out, opts=opts, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    clocks = clock_sampler_stop(cp, cf, clk_path, local)
    vg.sync_status()
    recs = D.profile()
    ms = reduce_max(ms, dist)
    ms_step = ms / args.steps
    value = whole_job_tflops(step_flops, args.steps, world, ms / 1e3)

    # the roofline kernel from the events recorded inside the timed region
    sust, burst, hbm, src = peaks()
    dom = [r for r in recs if r["kind"] == "conv3x3" and all(r[k] == v for k, v in DOMINANT.items())]
    dom_ms = sum(r["ms"] for r in dom) / max(1, len(dom))
    dom_flops = dom[0]["flops"] if dom else 0.0
    achieved = dom_flops / (dom_ms / 1e3) / 1e12 if dom else 0.0

    # per-stage summaries from separate decodes with events around every stage
    n_prof = 3
    for _ in range(n_prof):
        D.decode(z, out=out, opts=opts_all, workspace=ws)
    vg.sync_status()
    recs_all = D.profile()
    by = {}
    for r in recs_all:
        b = by.setdefault(r["kind"], {"ms": 0.0, "flops": 0.0, "bytes": 0.0, "launches": 0})
        b["ms"] += r["ms"]
        b["flops"] += r["flops"]
        b["bytes"] += r["bytes"]
        b["launches"] += r["launches"]
    stages = {}
    for k, b in by.items():
        e = {"ms_per_step": b["ms"] / n_prof, "launches_per_step": b["launches"] // n_prof}
        if b["flops"] > 0:
            e["tflops"] = b["flops"] / (b["ms"] / 1e3) / 1e12
        if b["bytes"] > 0:
            e["gbs"] = b["bytes"] / (b["ms"] / 1e3) / 1e9
        stages[k] = e
    conv_all = by.get("conv3x3", {"flops": 0.0, "ms": 1.0})
    # every decode launches the same kernels: the profiled decodes' count per decode x timed decodes
    launches = sum(r["launches"] for r in recs_all) // n_prof * args.steps

    # end to end through the host-buffer call (pinned host buffers)
    zh = torch.from_numpy(latent_channel_stats(rank, *LATENT)).pin_memory()
    oh = torch.empty((3, h0 * 8, w0 * 8), dtype=torch.float32).pin_memory()
    ws2 = torch.empty(D.workspace_bytes(h0, w0), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        D.decode_host(zh, oh, ws2)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        D.decode_host(zh, oh, ws2)
    torch.cuda.synchronize()
    t_e2e = time.perf_counter() - t0
    t_e2e = reduce_max(t_e2e, dist)
    e2e_val = whole_job_tflops(step_flops, args.steps, world, t_e2e)

    # The same decode replayed as a CUDA graph (no profile events in it).
    dg = D.graph(z, out, ws2)
    for _ in range(2):
        dg.launch()
    torch.cuda.synchronize()
    e4 = torch.cuda.Event(enable_timing=True)
    e5 = torch.cuda.Event(enable_timing=True)
    e4.record(stream)
    for _ in range(args.steps):
        dg.launch()
    e5.record(stream)
    torch.cuda.synchronize()
    vg.sync_status()
    ms_graph = e4.elapsed_time(e5) / args.steps
    del dg

    # The opt-in sub-pixel form of the up convs (it changes the rounding, so it is
    # reported beside the contract's number, not as it): device decodes, events.
    opts_sp = vg.Decoder.opts(subpixel=True)
    if D.workspace_bytes(h0, w0, opts_sp) > ws2.numel():
        ws2 = torch.empty(D.workspace_bytes(h0, w0, opts_sp), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        D.decode(z, out=out, opts=opts_sp, workspace=ws2)
    torch.cuda.synchronize()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        D.decode(z, out=out, opts=opts_sp, workspace=ws2)
    e3.record(stream)
    torch.cuda.synchronize()
    vg.sync_status()
    ms_sp = e2.elapsed_time(e3) / args.steps

    extras = extra_configs(D, dec) if rank == 0 and not args.no_extra_configs else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        flops_s, ts = cpu_oracle_sample(dec, h0=32, w0=32, steps=1)
        cpu = {"value": flops_s / sum(ts) / 1e12, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
               "sample": f"oracle (float64 numpy) decode of the same decoder on a 32x32 latent (256^2 frame), "
                         f"{flops_s / 1e12:.3f} TFLOP in {sum(ts):.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "latent": list(LATENT), "frame": [h0 * 8, w0 * 8],
                       "frames_per_gpu_per_step": 1, "parallelism": f"replicas{world}" if world > 1 else "none",
                       "l2": "no flush: the per-step working set (weights ~0.3 GB, activations > 2 GB) exceeds the "
                             "126 MB L2",
                       "guard_log2": 8},
            "decode_ms_per_frame": ms_step, "mp_per_s": (h0 * 8) * (w0 * 8) * world / (ms_step / 1e3) / 1e6,
            "decode_ms_per_frame_subpixel_up": ms_sp,
            "decode_ms_per_frame_graph": ms_graph,
            "frac_of_f16_peak": value / burst,
            "conv3x3_tflops": conv_all["flops"] / (conv_all["ms"] / 1e3) / 1e12,
            "step_tflop": step_flops / 1e12,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
                         "frac": achieved / burst, "traffic": traffic_from_profiles(),
                         "frac_of_sustained": achieved / sust,
                         "frac_of_nominal_dense_f16": achieved / NOMINAL_F16_TFLOPS,
                         "kernel": "conv_kernel (three-tap halo stages) 3x3, 1024^2 x 144 -> 144 "
                                   "(M=1048576, N=144, K=1296)",
                         "flops_per_launch": dom_flops, "launches_timed": len(dom),
                         "peak_kind": f"bf16 dense burst ({src}); the conv runs inside a ~14 ms step at the "
                                      f"maximum SM clock, like the burst measurement"},
            "stages": stages,
            "stages_from": "3 decodes after the timed region with CUDA events around every stage",
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": int(zh.numel() * 4),
                    "d2h_bytes_per_step": int(oh.numel() * 4), "ms_per_step": 1e3 * t_e2e / args.steps},
            "gpu_launches": launches,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "other_configs": extras,
            "pages_context": {"resident_decode_1024_s_rtx_pro_4000": [0.49, 0.61],
                              "resident_decode_2048_s_rtx_pro_4000": 1.84,
                              "resident_decode_1536x2752_s_rtx_pro_4000": 1.87},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
