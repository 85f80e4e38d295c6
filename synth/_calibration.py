# Written by oracle/calibrate_skew.py; do not edit by hand.
# Oracle router at T=4096: hottest expert load / mean load = 9.797
ZIPF_ALPHA = 0.0546875
