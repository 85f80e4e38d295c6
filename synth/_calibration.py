# Written by oracle/calibrate_skew.py; do not edit by hand.
# Oracle router at T=4096: hottest expert load / mean load = 10.500
ZIPF_ALPHA = 0.0625
