"""Command-line view of a swizzled tile layout.

    python -m xor_swizzle_movement_gb300 --rows 8 --cols 64 --esize 2 --bms 3,3,3

prints each element's swizzled offset and bank (swz_layout_text), then, when
a GPU is present, runs swz_bank_profile on the warp accesses that read each
column down the first 32 rows and prints their cost in passes (1 = free of
bank conflicts)."""
import argparse

from . import swz_bank_profile, swz_layout_text


def main():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--rows", type=int, default=8)
    p.add_argument("--cols", type=int, default=64)
    p.add_argument("--esize", type=int, default=2, help="element bytes (1, 2, 4, 8, 16)")
    p.add_argument("--bms", default="3,3,3", help="B,M,S in element units")
    a = p.parse_args()
    B, M, S = (int(v) for v in a.bms.split(","))
    text = swz_layout_text(a.rows, a.cols, a.esize, B, M, S)
    print(f"Swizzle<{B},{M},{S}> on a {a.rows} x {a.cols} tile of {a.esize}-byte elements "
          "(physical offset / bank):")
    print(text, end="")
    try:
        import torch
        gpu = torch.cuda.is_available()
    except ImportError:
        gpu = False
    if not gpu:
        print("(column-read bank profile: needs a GPU)")
        return
    offs = [[int(cell.split("/")[0]) for cell in line.split()] for line in text.splitlines()]
    lanes = min(a.rows, 32)
    pats = [[offs[r][c] * a.esize for r in range(lanes)] + [0] * (32 - lanes) for c in range(a.cols)]
    addrs = torch.tensor(pats, dtype=torch.int64).to(torch.int32).cuda()
    mask = torch.full((a.cols,), (1 << lanes) - 1 if lanes < 32 else -1, dtype=torch.int64)
    active = mask.to(torch.int32).cuda()
    ways = torch.empty(a.cols, dtype=torch.int32, device="cuda")
    wavefronts = torch.empty_like(ways)
    swz_bank_profile(addrs, active, a.cols, a.esize, ways, wavefronts)
    torch.cuda.synchronize()
    print(f"column reads down the first {lanes} rows, worst pass cost per column (swz_bank_profile):",
          ways.cpu().tolist())


if __name__ == "__main__":
    main()
