"""Run as a fresh process by test_gpu_layer.py: several threads make the very
first layer calls of the process at the same time, each on its own stream with
its own inputs and workspace, so the library's one-time per-device launch setup
races and the persistent grouped GEMMs of different calls share the GPU (each
gets whatever SMs are free; tiles are claimed in order by running CTAs, so no
grid waits for CTAs that have not started); every result must equal a later
single-threaded call."""
import sys
import threading

import torch

import grouped_gemm_softmax_gb300 as moe
import synth


def main(n_threads: int) -> int:
    cfgs = [synth.CONFIGS["tiny"], synth.CONFIGS["tiny"], synth.CONFIGS["mid"], synth.CONFIGS["tiny"]]
    jobs = []
    for i in range(n_threads):
        cfg = cfgs[i % len(cfgs)]
        shape = moe.Shape(T=cfg.T, d=cfg.d, E=cfg.E, top_k=cfg.k, ffn=cfg.F, num_segments=cfg.S)
        inp = synth.make_inputs(cfg, seed=10 + i, device="cuda")
        ws = moe.alloc_workspace(shape)
        out = [torch.empty(cfg.T // cfg.S, cfg.d, dtype=torch.bfloat16, device="cuda") for _ in range(cfg.S)]
        jobs.append((shape, inp, ws, out, torch.cuda.Stream()))
    torch.cuda.synchronize()
    start = threading.Barrier(n_threads)
    errors = []

    def run(job):
        shape, inp, ws, out, stream = job
        try:
            start.wait()
            with torch.cuda.stream(stream):
                for _ in range(3):
                    moe.layer_forward(shape, inp.x, inp.wr, inp.bias, inp.w1, inp.w3, inp.w2, out, ws,
                                      stream=stream)
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    torch.cuda.synchronize()
    if errors or any(t.is_alive() for t in threads):
        print("errors:", errors)
        return 1
    for shape, inp, ws, out, stream in jobs:
        if moe.last_device_status(ws, stream) != moe.MOE_OK:
            print("device status", moe.last_device_detail())
            return 1
        got = torch.cat(out, 0).clone()
        moe.layer_forward(shape, inp.x, inp.wr, inp.bias, inp.w1, inp.w3, inp.w2, out, ws)
        torch.cuda.synchronize()
        if not torch.equal(got.view(torch.int16), torch.cat(out, 0).view(torch.int16)):
            print("concurrent result differs from the single-threaded one")
            return 1
    print("ok")
    return 0


if __name__ == "__main__":
    sys.exit(main(int(sys.argv[1]) if len(sys.argv) > 1 else 4))
