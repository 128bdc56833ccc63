"""Small fixed cases for profiler captures: one dual-stream or single-stream block at the
1024x1024 shape (512 text + 4096 image tokens, hidden 3072), or the per-step modulation at
klein width (batch 1), run `--reps` times through the C ABI.  About 1 GB on the device for
a block (its GEMMs read more than the 129 MB L2); 341 MB of modulation weights for the
modulation.

    python -m diffusion_transformer_step_gb300.profile_case --block single --reps 2
    python -m diffusion_transformer_step_gb300.profile_case --block modulation --reps 3
    python -m diffusion_transformer_step_gb300.profile_case --block single --fp8 --reps 2

`--fp8` runs the block with every projection in e4m3 (per-row activation and per-output-channel
weight scales, the library's low-precision variant).
"""
import argparse

import torch

from diffusion_transformer_step_gb300 import build_lib, dit, synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--block", choices=["single", "dual", "modulation"], default="single")
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--fp8", action="store_true", help="every block projection in e4m3")
    args = ap.parse_args()
    build_lib.build()
    dev = "cuda"
    wl = synth.WORKLOADS["single_block_1024"]
    wd = wl.widths
    g = synth.generator(0, dev)
    if args.block == "modulation":
        W = dit.DeviceWeights(wd, {"mod": synth.mod_weights(wd, g, dev), "dual": [], "single": []}, device=dev)
        sigma = torch.full((1,), 0.75, dtype=torch.float32, device=dev)
        mod = torch.empty((1, 17 * wd.hidden), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
        for _ in range(args.reps):
            dit.dit_modulation(W.w, sigma, 1, mod, ws, ws.numel())
        st, where = dit.dit_sync_status(ws)
        assert st == dit.DIT_OK, f"device wait gave up at site {where:#x}"
        print(f"profile_case modulation x{args.reps}: ok")
        return
    if args.block == "dual":
        logical = {"dual": [(synth.stream_weights(wd, g, dev), synth.stream_weights(wd, g, dev))], "single": []}
    else:
        logical = {"dual": [], "single": [synth.single_weights(wd, g, dev)]}
    W = dit.DeviceWeights(wd, logical, device=dev, fp8="all" if args.fp8 else False)
    bi = synth.block_inputs(wl, 0, dev)
    shape = dit.make_shape(wl.batch, wl.n_txt, wl.n_img, wl.n_ref)
    ids = dit.dit_token_ids(shape, *wl.grid)
    N = wl.n_tokens
    rope = torch.empty((N, 64, 2), dtype=torch.float32, device=dev)
    dit.dit_rope_table(W.cfg, ids.to(dev), N, rope)
    nbytes = dit.dit_workspace_size(W.cfg, shape)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    fwd = dit.dit_dual_block_fwd if args.block == "dual" else dit.dit_single_block_fwd
    for _ in range(args.reps):
        fwd(W.w, 0, shape, bi["x"], bi["mod"], rope, ws, nbytes)
    st, where = dit.dit_sync_status(ws)
    assert st == dit.DIT_OK, f"device wait gave up at site {where:#x}"
    print(f"profile_case {args.block}{' e4m3' if args.fp8 else ''} x{args.reps}: ok")


if __name__ == "__main__":
    main()
