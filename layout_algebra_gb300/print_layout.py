"""Print the offset grid of rank-2 layouts:

    python -m layout_algebra_gb300.print_layout "(4,8):(1,4)" "((2,2),(2,2)):((1,4),(2,8))"
"""
import sys

from .layout import LayoutError, print_layout


def main(argv=None):
    args = sys.argv[1:] if argv is None else argv
    if not args:
        print(__doc__.strip())
        return 2
    for a in args:
        try:
            print(print_layout(a))
        except LayoutError as e:
            print("%s: %s" % (a, e))
            return 1
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
