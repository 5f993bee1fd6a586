"""One rank of the multi-process check of bench.py's host logic (launched by
tests/test_multiproc.py through torch.distributed.run with the gloo backend, no GPU)."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))

import bench  # noqa: E402


def main():
    world, rank, local, pg = bench.dist_setup(None)
    bench.barrier(pg)
    out = {
        "rank": rank, "world": world, "local": local,
        "max": bench.max_over_ranks(pg, 10.0 * (rank + 1)),
        "sum": bench.sum_over_ranks(pg, rank + 1),
    }
    bench.barrier(pg)
    with open(os.path.join(sys.argv[1], f"rank{rank}.json"), "w") as f:
        json.dump(out, f)
    pg.destroy_process_group()


if __name__ == "__main__":
    main()
