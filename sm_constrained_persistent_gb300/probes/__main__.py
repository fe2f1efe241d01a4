"""Builds and runs the measurement probes on cuda:0 (see the package docstring)."""
import sys

from . import PROBES, run


def main(argv):
    for name in (argv or PROBES):
        sys.stdout.write(run(name))
        sys.stdout.flush()


if __name__ == "__main__":
    main(sys.argv[1:])
