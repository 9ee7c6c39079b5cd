// residency.cu -- bounded HBM expert cache (placeholder translation unit).
